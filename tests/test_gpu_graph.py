"""The forward call captured in a CUDA graph (as a rollout engine captures its decode
step) and replayed on new inputs gives the eager call's bits."""
import pytest
import torch

from invariant_selected_token_gb300 import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,n_shards", [(1, 4), (64, 1), (300, 4)])
def test_linear_logprob_graph_replay(rlk, cuda_device, T, n_shards):
    H, V = 512, 20000
    batches = [WL.to_device(WL.small_case(T, H, V, seed=s), cuda_device) for s in (61, 62, 63)]
    W = batches[0].W
    eager = [rlk.linear_logprob(b.hidden, W, b.targets, None, n_shards) for b in batches]
    hidden = batches[0].hidden.clone()
    targets = batches[0].targets.clone()
    lp = torch.empty(T, dtype=torch.float32, device=cuda_device)
    lse = torch.empty_like(lp)
    ws = rlk.new_workspace(T, V, n_shards, cuda_device)
    s = torch.cuda.Stream(cuda_device)
    s.wait_stream(torch.cuda.current_stream(cuda_device))
    with torch.cuda.stream(s):  # the first call on the device does its set-up outside capture
        rlk.linear_logprob(hidden, W, targets, None, n_shards, lp, lse, ws, stream=s)
    torch.cuda.current_stream(cuda_device).wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rlk.linear_logprob(hidden, W, targets, None, n_shards, lp, lse, ws,
                           stream=torch.cuda.current_stream(cuda_device))
    for rep in range(2):
        for b, (e_lp, e_lse) in zip(batches, eager):
            hidden.copy_(b.hidden)
            targets.copy_(b.targets)
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(lp.view(torch.int32), e_lp.view(torch.int32)), rep
            assert torch.equal(lse.view(torch.int32), e_lse.view(torch.int32)), rep
