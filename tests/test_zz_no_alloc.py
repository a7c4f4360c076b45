"""rlk_linear_logprob_static_ws: the entry point for callers that cannot allocate.

Some callers have no way to hand the library a workspace: a rollout engine
that reserved nearly all device memory for its KV cache at start-up, or a
decode loop that cannot take the device-wide synchronisation cudaFree
implies.  rlk_linear_logprob_static_ws serves them from a scratch array
compiled into the library.  This test calls it through the C-ABI (ctypes,
no binding helper) twice in a row, on two different batches, and checks
each result against rlk_linear_logprob on the same inputs: within the
tolerance the parity tests use, and in fact bit for bit, since both run the
same kernels.  The second call also shows that what the first call left in
the shared scratch does not leak into the next result.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

TOL_LP = 1e-4
TOL_LSE_REL = 2e-5
STATIC_WS_BYTES = 16 << 20


def _static_ws_fn(lib):
    fn = lib.rlk_linear_logprob_static_ws
    P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.restype = i32
    fn.argtypes = [P, P, P, P, i64, i64, i64, i32, P, P, P, P]
    return fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_static(fn, dw, n_shards, status):
    T, H = dw.hidden.shape
    V = dw.W.shape[0]
    lp = torch.full((T,), float("nan"), dtype=torch.float32, device=dw.hidden.device)
    lse = torch.full((T,), float("nan"), dtype=torch.float32, device=dw.hidden.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dw.hidden.device).cuda_stream)
    rc = fn(_p(dw.hidden), _p(dw.W), _p(dw.targets), _p(dw.active), T, H, V, n_shards, _p(lp),
            _p(lse), _p(status), stream)
    return rc, lp, lse


def _compare(rlk, dw, n_shards, lp, lse):
    ref_lp, ref_lse = rlk.linear_logprob(dw.hidden, dw.W, dw.targets, dw.active, n_shards)
    torch.cuda.synchronize()
    a, b = lp.cpu().numpy(), ref_lp.cpu().numpy()
    c, d = lse.cpu().numpy(), ref_lse.cpu().numpy()
    assert np.all(np.isfinite(a)) and np.all(np.isfinite(c))
    assert np.abs(a.astype(np.float64) - b).max() <= TOL_LP
    assert (np.abs(c.astype(np.float64) - d) / np.maximum(np.abs(d), 1.0)).max() <= TOL_LSE_REL
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.array_equal(c.view(np.uint32), d.view(np.uint32))


def test_static_scratch_entry_point_matches_workspace_path(rlk, cuda_device):
    fn = _static_ws_fn(rlk.lib())
    status = rlk.new_status(cuda_device)
    first = WL.to_device(WL.small_case(300, 256, 5000, seed=41, n_shards=4, inactive_frac=0.1),
                         cuda_device)
    second = WL.to_device(WL.small_case(77, 512, 12345, seed=42, n_shards=2), cuda_device)
    rc1, lp1, lse1 = _call_static(fn, first, 4, status)
    rc2, lp2, lse2 = _call_static(fn, second, 2, status)
    assert rc1 == 0 and rc2 == 0
    torch.cuda.synchronize()
    rlk.raise_on_device_status(status)
    _compare(rlk, first, 4, lp1, lse1)
    _compare(rlk, second, 2, lp2, lse2)


def test_static_scratch_refuses_batches_beyond_its_size(rlk, cuda_device):
    fn = _static_ws_fn(rlk.lib())
    V, n = 151936, 4
    T_ok = 1
    while rlk.workspace_size(T_ok + 1, V, n) <= STATIC_WS_BYTES:
        T_ok += 1
    assert 1500 < T_ok < 2000
    W = torch.zeros((V, 64), dtype=torch.bfloat16, device=cuda_device)
    h = torch.zeros((T_ok + 1, 64), dtype=torch.bfloat16, device=cuda_device)
    tg = torch.zeros(T_ok + 1, dtype=torch.int32, device=cuda_device)
    out = torch.empty(T_ok + 1, dtype=torch.float32, device=cuda_device)
    stream = ctypes.c_void_p(torch.cuda.current_stream(cuda_device).cuda_stream)
    rc = fn(_p(h), _p(W), _p(tg), None, T_ok + 1, 64, V, n, _p(out), _p(out), None, stream)
    assert rc == 4  # RLK_ERR_WORKSPACE, nothing launched
    # a missing output is reported first, as rlk_linear_logprob reports it
    rc = fn(_p(h), _p(W), _p(tg), None, T_ok + 1, 64, V, n, None, _p(out), None, stream)
    assert rc == 1  # RLK_ERR_INVALID_ARG


def test_static_scratch_later_calls_take_no_device_memory(rlk, cuda_device):
    """After the first call on the device has loaded the scratch array, further calls leave
    the device's free memory exactly as it was: nothing is allocated per call."""
    fn = _static_ws_fn(rlk.lib())
    status = rlk.new_status(cuda_device)
    dw = WL.to_device(WL.small_case(200, 256, 7000, seed=43, n_shards=2), cuda_device)
    rc, _, _ = _call_static(fn, dw, 2, status)   # first call: loads the array if not yet loaded
    assert rc == 0
    lp = torch.empty(200, dtype=torch.float32, device=cuda_device)
    lse = torch.empty_like(lp)
    stream = ctypes.c_void_p(torch.cuda.current_stream(cuda_device).cuda_stream)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(cuda_device)
    for _ in range(3):
        rc = fn(_p(dw.hidden), _p(dw.W), _p(dw.targets), _p(dw.active), 200, 256, 7000, 2,
                _p(lp), _p(lse), _p(status), stream)
        assert rc == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(cuda_device)
    rlk.raise_on_device_status(status)
    assert free1 == free0, (free0, free1)
