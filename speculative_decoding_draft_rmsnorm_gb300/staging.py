"""Host-fed calls: a step's host-side inputs in one pinned buffer, moved to the device with one copy.

A caller whose inputs start on the host (tokens' rows, lengths, positions) would otherwise issue one
host-to-device copy per tensor, each paying the copy engine's fixed cost. Here every input gets an
aligned slice of one pinned host buffer and of one device buffer of the same layout; `upload()`
enqueues a single copy on the stream, after which the device views are ready for the library's
calls. Plumbing only: no arithmetic of the method lives here.
"""
from __future__ import annotations

import numpy as np

_ALIGN = 256  # every slice starts on a 256-byte boundary (TMA wants 16)


def _torch_dtype(dtype: np.dtype):
    import torch
    table = {np.dtype(np.uint16): torch.int16, np.dtype(np.int16): torch.int16, np.dtype(np.int32): torch.int32,
             np.dtype(np.int64): torch.int64, np.dtype(np.float32): torch.float32, np.dtype(np.uint8): torch.uint8}
    if np.dtype(dtype) not in table:
        raise TypeError(f"unsupported staging dtype {dtype}")
    return table[np.dtype(dtype)]


class HostStaging:
    """Named device views over one buffer filled from one pinned host buffer.

    arrays: name -> numpy array giving each input's shape and dtype (uint16 arrays are bf16 bit
    patterns and come out as torch.bfloat16 views). `fill(name, array)` writes an input on the
    host; `upload(stream)` copies the whole buffer; `views[name]` are the device tensors.
    """

    def __init__(self, arrays: dict, device="cuda"):
        import torch
        self.layout = {}
        off = 0
        for name, a in arrays.items():
            a = np.asarray(a)
            self.layout[name] = (off, a.nbytes, a.dtype, a.shape)
            off += (a.nbytes + _ALIGN - 1) // _ALIGN * _ALIGN
        self.nbytes = max(off, _ALIGN)
        self.host = torch.empty(self.nbytes, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.views = {}
        self._host_np = self.host.numpy()
        for name, (o, n, dt, shape) in self.layout.items():
            v = self.dev[o:o + n].view(_torch_dtype(dt)).view(shape)
            self.views[name] = v.view(torch.bfloat16) if np.dtype(dt) == np.uint16 else v
        for name, a in arrays.items():
            self.fill(name, a)

    def fill(self, name: str, array) -> None:
        o, n, dt, shape = self.layout[name]
        a = np.ascontiguousarray(array, dtype=dt)
        if a.shape != tuple(shape):
            raise ValueError(f"{name}: shape {a.shape}, staged as {tuple(shape)}")
        self._host_np[o:o + n] = a.reshape(-1).view(np.uint8)

    def upload(self, stream=None) -> None:
        import torch
        s = stream or torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self.dev.copy_(self.host, non_blocking=True)
