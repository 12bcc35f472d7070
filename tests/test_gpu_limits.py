"""Problem sizes at the far ends of what the forward accepts, against the fp64
oracle on sampled rows (tile edges of the first, middle and last heads plus
random rows): one head of 2^17 - 1 keys (1024 KV tiles, the last one ragged)
on each kernel family (head dimension 128 non-causal and causal on the
CTA-pair kernel, 64 on the one-CTA kernel), and more than 65535 heads of a
sequence shorter than one tile (tens of thousands of persistent-schedule
rounds per CTA). The bound is the stated one on the sampled rows
(parity_util.compare: 1e-2 per element, 1e-3 mean, 1e-3 on the LSE), and on
every row: finite values and O within its head's V column range (O is a
convex combination of V rows)."""
import numpy as np
import pytest

import attention_forward_flashattention_gb300 as fa
from attention_forward_flashattention_gb300 import inputs as I

from parity_util import bits_to_f64, compare, half_ulp, record, run_fa, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    torch.cuda.init()
    fa.build.build()
    fa.load_library()


def _check_all_rows(o_bits, lse, v_bits, w):
    """Every row finite, every O element inside its column's range over the
    head's keys (visible or not: a superset of the causal row's keys)."""
    vd = bits_to_f64(v_bits, w.dtype).reshape(w.B * w.H, w.N, w.d)
    od = bits_to_f64(o_bits, w.dtype).reshape(w.B * w.H, w.N, w.d)
    assert np.all(np.isfinite(od)) and np.all(np.isfinite(lse))
    lo, hi = vd.min(axis=1, keepdims=True), vd.max(axis=1, keepdims=True)
    slack = 1e-3 + half_ulp(od, w.dtype)
    assert np.all(od >= lo - slack) and np.all(od <= hi + slack)


def _sampled(oracle_mod, w, n_rows, seed, expect_cluster):
    info = fa.fa_query_launch(w.B, w.H, w.N, w.d, w.causal)
    assert info["cluster"] == expect_cluster
    q, k, v = I.qkv_bits(w)
    o, lse = run_fa(q, k, v, w.dtype, w.causal, w.scale)
    rows = sample_rows(w.B, w.H, w.N, n_rows, seed=seed)
    o_ref, l_ref = oracle_mod.attn_rows(q, k, v, w.dtype, w.causal, w.scale, rows)
    res = compare(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, l_ref, w.dtype)
    record(w.name, {k: x for k, x in res.items() if not k.startswith("_")}, rows=int(rows.size))
    assert res["ok"], {k: x for k, x in res.items() if not k.startswith("_")}
    _check_all_rows(o, lse, v, w)


LONG = [
    # N, d, dtype, causal, cluster of the kernel fa_fwd picks
    (131071, 128, "fp16", False, 2),
    (131071, 128, "bf16", True, 2),
    (131071, 64, "fp16", True, 1),
    (131071, 64, "bf16", False, 1),
]


@pytest.mark.parametrize("N,d,dtype,causal,cluster", LONG)
def test_one_long_head(oracle_mod, N, d, dtype, causal, cluster):
    w = I.custom(f"long_n{N}_d{d}_{dtype}_c{int(causal)}", 1, 1, N, d, dtype, causal,
                 seed_index=4100 + d + int(causal))
    _sampled(oracle_mod, w, 48, seed=41, expect_cluster=cluster)


MANY = [
    # B, H, N, d, dtype, causal, cluster
    (2, 33000, 9, 64, "fp16", True, 1),
    (1, 66000, 9, 128, "fp16", False, 2),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,cluster", MANY)
def test_many_short_heads(oracle_mod, B, H, N, d, dtype, causal, cluster):
    w = I.custom(f"heads_b{B}_h{H}_n{N}_d{d}", B, H, N, d, dtype, causal,
                 seed_index=4200 + d)
    _sampled(oracle_mod, w, 96, seed=42, expect_cluster=cluster)
