"""CUDA graphs: the forward (one-CTA and CTA-pair kernels), the 8-bit forward
and the backward captured once into a torch.cuda.CUDAGraph and replayed on new
input values give, bit for bit, what the same calls give when launched
directly. The calls only enqueue work on the given stream (tensor maps are
encoded on the host and passed by value as kernel parameters), so a replay
runs them on whatever the captured buffers hold."""
import pytest

import attention_forward_flashattention_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    torch.cuda.init()
    fa.build.build()
    fa.load_library()


def _fill(ts, seed):
    import torch
    g = torch.Generator(device="cuda:0").manual_seed(seed)
    for t in ts:
        if t.dtype == torch.uint8:   # e4m3 codes
            t.copy_(torch.randn(t.shape, device="cuda:0", generator=g)
                    .to(torch.float8_e4m3fn).view(torch.uint8))
        else:
            t.copy_(torch.randn(t.shape, device="cuda:0", generator=g).to(t.dtype))


def _capture(fn):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):      # warm-up outside the capture
        fn(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(torch.cuda.current_stream())
    return g


@pytest.mark.parametrize("B,H,N,d,dtype,causal,cluster", [
    (1, 6, 1000, 64, "bf16", True, 1),
    (2, 16, 2048, 128, "fp16", False, 2),
])
def test_forward_graph_replays_match_direct_launches(B, H, N, d, dtype, causal, cluster):
    import torch
    assert fa.fa_query_launch(B, H, N, d, causal)["cluster"] == cluster
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    q, k, v, o = (torch.empty(B, H, N, d, dtype=tdt, device="cuda:0") for _ in range(4))
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda:0")
    _fill((q, k, v), 1)
    g = _capture(lambda s: fa.attention_forward_into(q, k, v, o, lse, causal, None, s))
    for seed in (2, 3, 4):
        _fill((q, k, v), seed)
        g.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = fa.attention_forward(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert fa.fa_check(0) == fa.FA_OK


def test_fp8_forward_graph_replays_match_direct_launches():
    import torch
    B, H, N, d = 1, 4, 1500, 128
    q8, k8 = (torch.empty(B, H, N, d, dtype=torch.uint8, device="cuda:0") for _ in range(2))
    vt8 = torch.empty(B, H, d, 1504, dtype=torch.uint8, device="cuda:0")  # rows of 16-byte multiples
    ks = torch.rand(B, H, (N + 127) // 128, device="cuda:0") + 0.5
    o = torch.empty(B, H, N, d, dtype=torch.bfloat16, device="cuda:0")
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda:0")
    _fill((q8, k8, vt8), 5)
    g = _capture(lambda s: fa.attention_forward_fp8_into(q8, k8, vt8, o, lse, 0.8, ks, 1.2,
                                                         True, None, s))
    for seed in (6, 7):
        _fill((q8, k8, vt8), seed)
        g.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = fa.attention_forward_fp8(q8, k8, vt8, 0.8, ks, 1.2, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert fa.fa_check(0) == fa.FA_OK


def test_backward_graph_replays_match_direct_launches():
    import torch
    B, H, N, d = 1, 4, 1100, 128
    q, k, v, do = (torch.empty(B, H, N, d, dtype=torch.float16, device="cuda:0")
                   for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device="cuda:0")
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda:0")
    scale = d ** -0.5

    def step(s):   # forward then backward, as in a training step
        fa.attention_forward_into(q, k, v, o, lse, True, scale, s)
        rc = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                       lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                       ws.data_ptr(), B, H, N, d, True, scale, fa.FA_DTYPE_FP16,
                       int(s.cuda_stream))
        assert rc == fa.FA_OK, fa.status_string(rc)

    _fill((q, k, v, do), 8)
    g = _capture(step)
    for seed in (9, 10):
        _fill((q, k, v, do), seed)
        g.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = fa.attention_forward(q, k, v, causal=True, scale=scale)
        ref = fa.attention_backward(q, k, v, o_ref, l_ref, do, causal=True, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
        assert all(torch.equal(a, b) for a, b in zip((dq, dk, dv), ref))
    assert fa.fa_check(0) == fa.FA_OK
