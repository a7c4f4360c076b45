"""The forward call captured in a CUDA graph (as a rollout engine captures its decode
step) and replayed on new inputs gives the eager call's bits; so do both backward paths
(a training step captures them), whose split sum forks onto a second stream and joins
back inside the graph."""
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


@pytest.mark.parametrize("saved", [False, True])
def test_backward_graph_replay(rlk, cuda_device, saved):
    """The backward (both gradients: its split sum forks onto the library's side stream
    and joins back) captured in a CUDA graph and replayed on new inputs gives the eager
    call's bits; with `saved`, the saving forward and the backward from its logits."""
    T, H, V = 200, 256, 3000
    batches = [WL.to_device(WL.small_case(T, H, V, seed=s, w_std=0.05), cuda_device)
               for s in (71, 72)]
    W = batches[0].W
    g_in = torch.linspace(-1.0, 1.0, T, dtype=torch.float32, device=cuda_device)

    def run(b_hidden, b_targets, out_dh, out_dW, stream, logits=None, ws_f=None, ws_b=None):
        if saved:
            _, lse, _ = rlk.linear_logprob_save_logits(b_hidden, W, b_targets, logits=logits,
                                                       workspace=ws_f, stream=stream)
            rlk.linear_logprob_backward_from_logits(logits, b_hidden, W, b_targets, g_in, lse,
                                                    grad_hidden=out_dh, grad_W=out_dW,
                                                    workspace=ws_b, stream=stream)
        else:
            _, lse = rlk.linear_logprob(b_hidden, W, b_targets, workspace=ws_f, stream=stream)
            rlk.linear_logprob_backward(b_hidden, W, b_targets, g_in, lse, grad_hidden=out_dh,
                                        grad_W=out_dW, workspace=ws_b, stream=stream)

    cur = torch.cuda.current_stream(cuda_device)
    eager = []
    for b in batches:
        dh = torch.empty((T, H), dtype=torch.float32, device=cuda_device)
        dW = torch.empty((V, H), dtype=torch.float32, device=cuda_device)
        run(b.hidden, b.targets, dh, dW, cur,
            logits=torch.empty((T, (V + 3) // 4 * 4), dtype=torch.float32, device=cuda_device))
        eager.append((dh, dW))
    hidden = batches[0].hidden.clone()
    targets = batches[0].targets.clone()
    dh = torch.empty((T, H), dtype=torch.float32, device=cuda_device)
    dW = torch.empty((V, H), dtype=torch.float32, device=cuda_device)
    logits = torch.empty((T, (V + 3) // 4 * 4), dtype=torch.float32, device=cuda_device)
    ws_f = rlk.new_workspace(T, V, 1, cuda_device)
    ws_b = torch.empty(rlk.backward_workspace_size(T, H, V), dtype=torch.uint8, device=cuda_device)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(hidden, targets, dh, dW, torch.cuda.current_stream(cuda_device), logits, ws_f, ws_b)
    for rep in range(2):
        for b, (e_dh, e_dW) in zip(batches, eager):
            hidden.copy_(b.hidden)
            targets.copy_(b.targets)
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(dh.view(torch.int32), e_dh.view(torch.int32)), rep
            assert torch.equal(dW.view(torch.int32), e_dW.view(torch.int32)), rep
