"""fa_fwd_host: the forward on host buffers with chunked copy / compute
overlap gives, bit for bit, what the device entry point gives on the same
inputs (each row's arithmetic does not depend on how the heads are chunked),
for one chunk and several uneven ones (the first and last half size), odd N
(per-chunk LSE blocks padded to 16 bytes), page-locked and pageable host
memory; plus sampled rows against the fp64 oracle."""
import numpy as np
import pytest

import attention_forward_flashattention_gb300 as fa
from attention_forward_flashattention_gb300 import inputs as I

from parity_util import bits_to_f64, half_ulp, sample_rows, to_bits, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    torch.cuda.init()
    fa.build.build()
    fa.load_library()


def _host_tensors(x, dtype, pin):
    import torch
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    t = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(tdt) for a in x]
    return [a.pin_memory() for a in t] if pin else t


CASES = [
    # B, H, N, d, dtype, causal, pinned
    (2, 3, 300, 128, "fp16", True, True),     # one chunk
    (1, 701, 255, 64, "bf16", False, True),   # five uneven chunks (4 + 1), odd N
    (4, 16, 4096, 128, "fp16", False, True),  # the default workload's shape: seven chunks
    (1, 701, 255, 64, "fp16", True, False),   # pageable host memory
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,pinned", CASES)
def test_host_matches_device_path(B, H, N, d, dtype, causal, pinned):
    import torch
    w = I.custom("host", B, H, N, d, dtype, causal, seed_index=700 + H + N)
    x = I.qkv_bits(w)
    q, k, v = _host_tensors(x, dtype, pinned)
    o_h, lse_h = fa.attention_forward_host(q, k, v, causal=causal, scale=w.scale)
    assert fa.fa_check(0) == fa.FA_OK
    qd, kd, vd = (to_device(a, dtype) for a in x)
    o_d, lse_d = fa.attention_forward(qd, kd, vd, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(o_h), to_bits(o_d))
    assert np.array_equal(lse_h.numpy(), lse_d.cpu().numpy())


def test_host_sampled_rows_match_oracle(oracle_mod):
    w = I.custom("hostref", 1, 701, 255, 64, "bf16", True, seed_index=1701)
    x = I.qkv_bits(w)
    q, k, v = _host_tensors(x, "bf16", True)
    o_h, lse_h = fa.attention_forward_host(q, k, v, causal=True, scale=w.scale)
    rows = sample_rows(w.B, w.H, w.N, 64, seed=5)
    o_ref, l_ref = oracle_mod.attn_rows(*x, "bf16", True, w.scale, rows)
    got = bits_to_f64(to_bits(o_h).reshape(-1, w.d)[rows], "bf16")
    assert np.all(np.abs(got - o_ref) <= 1e-2 + half_ulp(o_ref, "bf16"))
    assert np.max(np.abs(lse_h.numpy().reshape(-1)[rows] - l_ref)) <= 1e-3


def test_host_workspace_too_small_is_rejected():
    import torch
    q = torch.zeros((1, 2, 128, 64), dtype=torch.float16)
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 128), dtype=torch.float32)
    ws = torch.empty(fa.fa_fwd_host_workspace_size(1, 2, 128, 64) - 16, dtype=torch.uint8,
                     device="cuda:0")
    with pytest.raises(fa.FaError):
        fa.attention_forward_host_into(q, q, q, o, lse, ws)
