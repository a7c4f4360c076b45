"""No kernel writes outside the buffers it is given.

Every output and workspace buffer is carved out of a larger allocation whose
margins hold a sentinel byte pattern; after each call the margins must be
unchanged (a light stand-in for a memory checker, which is not available on
the test machines).
"""
import numpy as np
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

PAD = 4096  # bytes of canary on each side


class Canary:
    def __init__(self, nbytes, dev):
        self.n = nbytes
        self.buf = torch.full((nbytes + 2 * PAD,), 0xA5, dtype=torch.uint8, device=dev)

    def view(self, dtype, shape):
        return self.buf[PAD:PAD + self.n].view(dtype).view(shape)

    def intact(self):
        b = self.buf.cpu().numpy()
        return bool(np.all(b[:PAD] == 0xA5) and np.all(b[PAD + self.n:] == 0xA5))


@pytest.mark.parametrize("T,H,V,n", [(1, 64, 1, 1), (37, 128, 1000, 4), (300, 256, 5000, 8),
                                     (130, 512, 2047, 2)])
def test_forward_shard_materialised_backward_rmsnorm_stay_in_bounds(rlk, cuda_device, T, H, V, n):
    w = WL.to_device(WL.small_case(T, H, V, seed=T + V, inactive_frac=0.2 if T > 4 else 0),
                     cuda_device)
    f32 = torch.float32
    lp, lse = Canary(4 * T, cuda_device), Canary(4 * T, cuda_device)
    ws = Canary(rlk.workspace_size(T, V, n), cuda_device)
    rlk.linear_logprob(w.hidden, w.W, w.targets, w.active, n, lp.view(f32, (T,)),
                       lse.view(f32, (T,)), ws.view(torch.uint8, (ws.n,)))
    torch.cuda.synchronize()
    assert lp.intact() and lse.intact() and ws.intact()

    vb, ve = rlk.shard_range(V, n, n - 1)
    part = Canary(16 * T, cuda_device)
    sws = Canary(rlk.workspace_size(T, ve - vb, 1), cuda_device)
    rlk.linear_logprob_shard(w.hidden, w.W[vb:ve], w.targets, w.active, V, n, n - 1,
                             part.view(torch.int32, (T, 4)), sws.view(torch.uint8, (sws.n,)))
    torch.cuda.synchronize()
    assert part.intact() and sws.intact()

    L = rlk.debug_logits(w.hidden, w.W)
    out = Canary(4 * T * V, cuda_device)
    mws = Canary(rlk.workspace_size(T, V, 1), cuda_device)
    olse = Canary(4 * T, cuda_device)
    rlk.log_softmax(L, w.active, out.view(f32, (T, V)), olse.view(f32, (T,)),
                    mws.view(torch.uint8, (mws.n,)))
    torch.cuda.synchronize()
    assert out.intact() and mws.intact() and olse.intact()

    g = torch.ones(T, device=cuda_device)
    dh, dW = Canary(4 * T * H, cuda_device), Canary(4 * V * H, cuda_device)
    bws = Canary(rlk.backward_workspace_size(T, H, V), cuda_device)
    _, lse_t = rlk.linear_logprob(w.hidden, w.W, w.targets, w.active, 1)
    rlk.linear_logprob_backward(w.hidden, w.W, w.targets, g, lse_t, w.active, True, True,
                                dh.view(f32, (T, H)), dW.view(f32, (V, H)),
                                bws.view(torch.uint8, (bws.n,)))
    torch.cuda.synchronize()
    assert dh.intact() and dW.intact() and bws.intact()

    gamma = torch.ones(H, dtype=torch.bfloat16, device=cuda_device)
    y, ro = Canary(2 * T * H, cuda_device), Canary(2 * T * H, cuda_device)
    rlk.rmsnorm(w.hidden, gamma, 1e-6, w.hidden, True, y.view(torch.bfloat16, (T, H)),
                ro.view(torch.bfloat16, (T, H)))
    torch.cuda.synchronize()
    assert y.intact() and ro.intact()
