"""The differentiable wrapper `attention`: its output and the gradients
autograd produces are, bit for bit, what attention_forward and
attention_backward give for the same inputs and output gradient (the wrapper
only routes the saved q, k, v, O and LSE to fa_bwd), for contiguous inputs and
for [B, N, H, d] storage passed as transposed views."""
import pytest

import attention_forward_flashattention_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    torch.cuda.init()
    fa.build.build()
    fa.load_library()


@pytest.mark.parametrize("B,H,N,d,dtype,causal,bnhd", [
    (1, 4, 700, 128, "fp16", True, False),
    (2, 3, 513, 64, "bf16", False, False),
    (2, 4, 640, 128, "bf16", True, True),
])
def test_autograd_matches_direct_calls(B, H, N, d, dtype, causal, bnhd):
    import torch
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    g = torch.Generator(device="cuda:0").manual_seed(B * 1000 + N)
    base = [torch.randn(B, H, N, d, device="cuda:0", generator=g).to(tdt) for _ in range(3)]
    w = torch.randn(B, H, N, d, device="cuda:0", generator=g)
    if bnhd:   # [B, N, H, d] storage seen as [B, H, N, d]
        leaves = [t.transpose(1, 2).contiguous().requires_grad_(True) for t in base]
        q, k, v = (t.transpose(1, 2) for t in leaves)
    else:
        leaves = [t.clone().requires_grad_(True) for t in base]
        q, k, v = leaves
    o = fa.attention(q, k, v, causal=causal)
    (o.float() * w).sum().backward()
    o_ref, lse_ref = fa.attention_forward(*base, causal=causal)
    dq, dk, dv = fa.attention_backward(*base, o_ref, lse_ref, w.to(tdt), causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o.detach(), o_ref)
    grads = [t.grad.transpose(1, 2) if bnhd else t.grad for t in leaves]
    for got, ref in zip(grads, (dq, dk, dv)):
        assert torch.equal(got, ref)
    assert fa.fa_check(0) == fa.FA_OK
