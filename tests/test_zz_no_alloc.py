"""The allocation-free sparse-MLA entry point (hs_sparse_mla_fwd_static) against the regular one.

hs_sparse_mla_fwd_static serves callers that cannot allocate device memory (their memory belongs
to another allocator, or they run where an allocation may not happen): its split-work scratch is
a fixed array inside the library instead of a caller workspace. Called through the C ABI twice in
a row with different inputs (the second call runs on whatever the first left in the shared
array), its output must match hs_sparse_mla_fwd with a caller workspace on the same inputs.
This file is collected last on purpose: a failure here leaves every other test already run.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import dsa_sparse_mla_gb300 as hs
from dsa_sparse_mla_gb300 import hs_check_flag, hs_sparse_mla_fwd, hs_sparse_mla_workspace_size, inputs

from parity import MLA_RTOL

pytestmark = pytest.mark.gpu


def _inputs(T, H, k, n, seed):
    st = inputs.Stream(seed)
    kv = inputs.pack_kv_rows(st.sub("l").normal((n, 512)), st.sub("r").normal((n, 64)))
    q = inputs.bf16_bits(st.sub("q").normal((T, H, 576)))
    rng = np.random.default_rng(seed)
    idx = rng.integers(0, n, (T, k)).astype(np.int32)
    idx[1, k // 3:] = -1                                   # a ragged query
    return (torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16), torch.from_numpy(kv).cuda(),
            torch.from_numpy(idx).cuda())


def _static_call(q, kv, idx, scale, out, lse, err):
    """hs_sparse_mla_fwd_static through the C ABI (ctypes, no binding helper)."""
    T, H, _ = q.shape
    a = hs._MlaArgs(T, H, idx.shape[1], q.data_ptr(), kv.data_ptr(), kv.shape[0], idx.data_ptr(), None, 0, None,
                    float(scale), out.data_ptr(), lse.data_ptr(), err.data_ptr(), None, 0)
    st = hs.load().hs_sparse_mla_fwd_static(ctypes.byref(a), torch.cuda.current_stream().cuda_stream)
    assert st == 0, hs.load().hs_last_error().decode()


def test_static_scratch_matches_workspace_call_twice():
    torch.cuda.set_device(0)
    H, k, n, scale = 64, 2048, 6000, 1 / math.sqrt(576)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for call, (T, seed) in enumerate([(40, 101), (37, 202)]):
        # fewer queries than 3/4 of one wave: the split-work path, and so the scratch, is taken
        assert 4 * T < 3 * sms, "this device has too few SMs for the split path at T = %d" % T
        q, kv, idx = _inputs(T, H, k, n, seed)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out_s = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse_s = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
        _static_call(q, kv, idx, scale, out_s, lse_s, err)
        torch.cuda.synchronize()
        # nothing allocated: not through torch, and (after the first call, which may load the
        # library's device code and its static array) not on the device at all
        assert torch.cuda.memory_allocated() == alloc0
        if call > 0:
            assert torch.cuda.mem_get_info()[0] == free0
        out_w = torch.empty_like(out_s)
        lse_w = torch.empty_like(lse_s)
        ws = torch.empty(hs_sparse_mla_workspace_size(H), dtype=torch.uint8, device="cuda")
        hs_sparse_mla_fwd(q, kv, idx, scale, out_w, err, lse=lse_w, workspace=ws)
        assert hs_check_flag(err) == 0, "call %d set the device error flag" % call
        g, r = out_s.float(), out_w.float()
        rel = ((g - r).abs().amax(-1) / r.abs().amax(-1).clamp_min(1e-6)).max().item()
        assert rel <= MLA_RTOL, "call %d: normwise difference %.3e" % (call, rel)
        d = ((lse_s - lse_w).abs() / lse_w.abs().clamp_min(1.0)).max().item()
        assert d <= MLA_RTOL, "call %d: lse difference %.3e" % (call, d)
