"""CUDA-graph capture of the library's launches.  The routing + expert-block forward (the
large-batch path, whose per-token quantisation runs on the library's side stream between
an event fork and join, and the decode-size path, a chain of programmatic dependent
launches) and the per-tensor quantiser (zeroing, amax and encode as a programmatic chain)
are captured once and replayed: every replay equals the eager launches bit for bit, and a
replay after the inputs were overwritten in place equals an eager run on the new inputs
(the graph reads the buffers, not the values seen at capture)."""
import pytest
import torch

from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Warm up on a side stream (as torch asks before a capture), then capture fn()."""
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.fixture(scope="module")
def moe_setup(cuda_lib):
    L = cuda_lib
    shape = S.WORKLOADS["gateup"]
    x_h, logits_h, w13_h, w2_h = S.moe_inputs(shape, seed=5)
    dev = torch.device("cuda", 0)
    pw = L.moe_prepare_weights(w13_h.to(dev), w2_h.to(dev))
    pt = L.moe_prepare_weights_backward(w13_h.to(dev), w2_h.to(dev))
    return L, shape, x_h, logits_h, pw, pt, dev


@pytest.mark.parametrize("T", [8, 2048])   # decode-size path (T*k <= 1024) and the large path
def test_forward_replays_in_a_cuda_graph(moe_setup, T):
    L, shape, x_h, logits_h, pw, _, dev = moe_setup
    k, H = shape.k, shape.H
    x = x_h[:T].contiguous().to(dev)
    logits = logits_h[:T].contiguous().to(dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws = L.moe_forward_workspace(T, k, pw, dev)

    def step():
        L.moe_route_topk(logits, k, True, out=(ids, w))
        L.moe_expert_forward(x, ids, w, pw, out=out, workspace=ws)

    step()
    torch.cuda.synchronize()
    ref_ids, ref_w, ref_out = ids.clone(), w.clone(), out.clone()
    g = _capture(step)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids) and torch.equal(w, ref_w)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    # new values in the captured input buffers: the replay follows them
    x.copy_(x_h[T:2 * T].to(dev))
    logits.copy_(logits_h[T:2 * T].to(dev))
    g.replay()
    torch.cuda.synchronize()
    got_ids, got_w, got_out = ids.clone(), w.clone(), out.clone()
    step()
    torch.cuda.synchronize()
    assert torch.equal(got_ids, ids) and torch.equal(got_w, w)
    assert torch.equal(got_out.view(torch.int16), out.view(torch.int16))
    assert not torch.equal(got_out.view(torch.int16), ref_out.view(torch.int16))
    assert L.nvfp4_status_check() == 0


def test_learner_step_replays_in_a_cuda_graph(moe_setup):
    """Routing, the forward and the W4A4 backward (stochastic rounding, fixed seed) of a
    1024-token batch as one graph."""
    L, shape, x_h, logits_h, pw, pt, dev = moe_setup
    T, k, H = 1024, shape.k, shape.H
    x = x_h[:T].contiguous().to(dev)
    logits = logits_h[:T].contiguous().to(dev)
    dout = S.randn_bf16((T, H), 1e-3, seed=9).to(dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    fws = L.moe_forward_workspace(T, k, pw, dev)
    bws = L.moe_backward_workspace(T, k, pw, dev)
    grads = (torch.empty(T, H, dtype=torch.bfloat16, device=dev), torch.empty(T, k, dtype=torch.float32, device=dev),
             torch.empty(pw.E, 2 * pw.I, H, dtype=torch.float32, device=dev),
             torch.empty(pw.E, H, pw.I, dtype=torch.float32, device=dev))

    def step():
        L.moe_route_topk(logits, k, True, out=(ids, w))
        L.moe_expert_forward(x, ids, w, pw, out=out, workspace=fws)
        L.moe_expert_backward(dout, x, w, pw, pt, fws, seed=21, out=grads, workspace=bws)

    def bits(t):
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)

    step()
    torch.cuda.synchronize()
    ref = [bits(t).clone() for t in (out,) + grads]
    g = _capture(step)
    for t in grads:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip([bits(t) for t in (out,) + grads], ref):
        assert torch.equal(a, b)
    dout.copy_(S.randn_bf16((T, H), 1e-3, seed=10).to(dev))
    g.replay()
    torch.cuda.synchronize()
    got = [bits(t).clone() for t in (out,) + grads]
    step()
    torch.cuda.synchronize()
    for a, b in zip(got, [bits(t) for t in (out,) + grads]):
        assert torch.equal(a, b)
    assert not torch.equal(got[1], ref[1])   # dx follows the new gradient
    assert L.nvfp4_status_check() == 0


@pytest.mark.parametrize("mode,rounding", [("tensor", "rne"), ("tensor", "sr"), ("row", "rne")])
def test_quantiser_replays_in_a_cuda_graph(cuda_lib, mode, rounding):
    L = cuda_lib
    dev = torch.device("cuda", 0)
    rows, cols = 1024, 2048
    x = S.outlier_channels_bf16(rows, cols, seed=3).to(dev)
    m = L.SCALE_PER_TENSOR if mode == "tensor" else L.SCALE_PER_ROW
    r = L.ROUND_RNE if rounding == "rne" else L.ROUND_STOCHASTIC
    codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(max(L.nvfp4_sf_bytes(rows, cols), 16), dtype=torch.uint8, device=dev)
    gs = torch.empty(rows, dtype=torch.float32, device=dev)
    ws = torch.empty(int(L.load().nvfp4_workspace_size(L.OP_QUANTIZE, rows, cols, 0, 0, 0)), dtype=torch.uint8,
                     device=dev)

    def q():
        L.nvfp4_quantize(x, m, r, seed=11, out=(codes, sf, gs), workspace=ws)

    q()
    torch.cuda.synchronize()
    ref = (codes.clone(), sf.clone(), gs.clone())
    g = _capture(q)
    codes.zero_()
    sf.zero_()
    g.replay()
    torch.cuda.synchronize()
    n_g = 1 if mode == "tensor" else rows
    assert torch.equal(codes, ref[0]) and torch.equal(sf, ref[1]) and torch.equal(gs[:n_g], ref[2][:n_g])
    # four times the values: the captured launches read the new ones (g follows; the codes
    # and block scales are invariant under a power-of-two factor)
    x.mul_(4.0)
    g.replay()
    torch.cuda.synchronize()
    got = (codes.clone(), sf.clone(), gs.clone())
    q()
    torch.cuda.synchronize()
    assert torch.equal(got[0], codes) and torch.equal(got[1], sf) and torch.equal(got[2][:n_g], gs[:n_g])
    assert torch.equal(got[2][:n_g], ref[2][:n_g] * 4.0)
    assert L.nvfp4_status_check() == 0
