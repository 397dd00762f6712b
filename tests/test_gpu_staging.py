"""The host-input staging buffer: one copy brings every input, each view holds its array's bits."""
from __future__ import annotations

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_one_upload_brings_every_input():
    import torch
    from speculative_decoding_draft_rmsnorm_gb300.staging import HostStaging
    rng = np.random.default_rng(0)
    arrays = {"a": rng.integers(0, 1 << 16, (37, 3, 8), dtype=np.uint64).astype(np.uint16),
              "b": rng.integers(-5, 5, 13).astype(np.int32),
              "c": rng.integers(0, 1 << 40, (2, 5)).astype(np.int64)}
    st = HostStaging(arrays)
    st.upload()
    torch.cuda.synchronize()
    assert st.views["a"].dtype == torch.bfloat16 and tuple(st.views["a"].shape) == (37, 3, 8)
    assert np.array_equal(st.views["a"].view(torch.int16).cpu().numpy().view(np.uint16), arrays["a"])
    assert np.array_equal(st.views["b"].cpu().numpy(), arrays["b"])
    assert np.array_equal(st.views["c"].cpu().numpy(), arrays["c"])
    for v in st.views.values():
        assert v.data_ptr() % 256 == 0
    # new host values, one more upload
    st.fill("b", arrays["b"] + 100)
    st.upload()
    torch.cuda.synchronize()
    assert np.array_equal(st.views["b"].cpu().numpy(), arrays["b"] + 100)
