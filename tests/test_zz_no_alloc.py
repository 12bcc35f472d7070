"""The allocation-free entry point, fa_fwd_noalloc.

It exists for callers that cannot allocate device memory (their allocator owns
all of HBM, or they must never call cudaMalloc / cudaFree while running): it
runs the same kernel as fa_fwd with the kernel's scratch (one status word) in
a fixed array inside the library. This test calls it through the C ABI twice
in a row and checks that both results equal fa_fwd's bit for bit (the same
deterministic kernel on the same inputs), and that fa_check, which reads the
allocation-free status word too, reports no timeout. It must pass alone in a
fresh process and after the other tests; the file name makes pytest collect
it last.
"""
import numpy as np
import pytest

import attention_forward_flashattention_gb300 as fa
from attention_forward_flashattention_gb300 import inputs as I

from parity_util import to_bits, to_device

pytestmark = pytest.mark.gpu


def _run(entry, q, k, v, w):
    import torch
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device=q.device)
    rc = entry(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
               w.B, w.H, w.N, w.d, w.causal, w.scale,
               fa.FA_DTYPE_BF16 if w.dtype == "bf16" else fa.FA_DTYPE_FP16,
               int(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_OK, fa.status_string(rc)
    torch.cuda.synchronize()
    return to_bits(o), lse.cpu().numpy()


@pytest.mark.parametrize("B,H,N,d,dtype,causal", [
    (2, 3, 1000, 128, "bf16", True),
    (1, 4, 640, 64, "fp16", False),
])
def test_noalloc_matches_fa_fwd_twice(B, H, N, d, dtype, causal):
    import torch
    torch.cuda.init()
    fa.build.build()
    fa.load_library()
    w = I.custom("noalloc", B, H, N, d, dtype, causal, seed_index=500 + d)
    qb, kb, vb = I.qkv_bits(w)
    q, k, v = (to_device(x, dtype) for x in (qb, kb, vb))
    sh = int(torch.cuda.current_stream().cuda_stream)
    o_ref, l_ref = _run(fa.fa_fwd, q, k, v, w)
    assert fa.fa_check(sh) == fa.FA_OK
    for _ in range(2):
        o, lse = _run(fa.fa_fwd_noalloc, q, k, v, w)
        assert np.array_equal(o, o_ref)
        assert np.array_equal(lse.view(np.uint32), l_ref.view(np.uint32))
        assert fa.fa_check(sh) == fa.FA_OK


def test_noalloc_rejects_bad_arguments():
    import torch
    torch.cuda.init()
    fa.load_library()
    x = torch.zeros((1, 1, 128, 96), dtype=torch.float16, device="cuda:0")
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device="cuda:0")
    p = x.data_ptr()
    assert fa.fa_fwd_noalloc(p, p, p, p, lse.data_ptr(), 1, 1, 128, 96, 0, 0.1, 0, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_noalloc(p, p, p, p, 0, 1, 1, 128, 64, 0, 0.1, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_noalloc(p, p, p, p, lse.data_ptr(), 1, 1, (1 << 30) + 1, 64, 0, 0.1, 0, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_noalloc(p, p, p, p, lse.data_ptr(), 0, 1, 128, 64, 0, 0.1, 0, 0) == fa.FA_ERR_INVALID_ARG
