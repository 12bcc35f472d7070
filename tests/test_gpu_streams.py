"""Calls on several streams at once. Forward calls (the one-CTA and the CTA-pair
kernel), an 8-bit forward and a backward, enqueued on four streams and running
concurrently, give bit for bit what the same calls give one after another on
the default stream: the library keeps no per-call device state beyond the
status word and the clock record, which only accumulate. And a backward on a
side stream keeps its workspace while its kernels run, even when the caller's
next allocations on the default stream ask for blocks of the same size."""
import pytest

import attention_forward_flashattention_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    torch.cuda.init()
    fa.build.build()
    fa.load_library()


def _inputs(B, H, N, d, dtype, seed):
    import torch
    g = torch.Generator(device="cuda:0").manual_seed(seed)
    return [torch.randn(B, H, N, d, device="cuda:0", generator=g).to(dtype) for _ in range(3)]


def _calls():
    """Four independent calls, each a function of an optional stream that
    returns its output tensors."""
    import torch
    q1, k1, v1 = _inputs(1, 8, 2000, 64, torch.bfloat16, 1)       # one-CTA, d = 64, causal
    q2, k2, v2 = _inputs(2, 16, 2048, 128, torch.float16, 2)      # CTA pairs
    assert fa.fa_query_launch(2, 16, 2048, 128, False)["cluster"] == 2
    g = torch.Generator(device="cuda:0").manual_seed(3)
    q8, k8 = (torch.randn(1, 4, 1024, 128, device="cuda:0", generator=g)
              .to(torch.float8_e4m3fn).view(torch.uint8) for _ in range(2))
    vt8 = (torch.randn(1, 4, 128, 1024, device="cuda:0", generator=g)
           .to(torch.float8_e4m3fn).view(torch.uint8))
    ks = torch.rand(1, 4, 8, device="cuda:0", generator=g) + 0.5
    q4, k4, v4 = _inputs(1, 4, 1024, 128, torch.float16, 4)       # backward
    o4, l4 = fa.attention_forward(q4, k4, v4, causal=True)
    do4 = torch.randn(q4.shape, device="cuda:0", generator=g).to(torch.float16)
    torch.cuda.synchronize()
    return [
        lambda s: fa.attention_forward(q1, k1, v1, causal=True, stream=s),
        lambda s: fa.attention_forward(q2, k2, v2, stream=s),
        lambda s: fa.attention_forward_fp8(q8, k8, vt8, 0.9, ks, 1.1, stream=s),
        lambda s: fa.attention_backward(q4, k4, v4, o4, l4, do4, causal=True, stream=s),
    ]


def _same(a, b):
    import torch
    return all(torch.equal(x, y) for x, y in zip(a, b))


def test_concurrent_streams_match_sequential_bits():
    import torch
    calls = _calls()
    ref = []
    for c in calls:
        ref.append([t.clone() for t in c(None)])
        torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in calls]
    outs = [[] for _ in calls]
    main = torch.cuda.current_stream()
    for s in streams:
        s.wait_stream(main)
    for _ in range(3):
        for i, (c, s) in enumerate(zip(calls, streams)):
            outs[i].append(c(s))
    torch.cuda.synchronize()
    for i, r in enumerate(ref):
        for got in outs[i]:
            assert _same(got, r), f"call {i}"
    assert fa.fa_check(0) == fa.FA_OK


def test_side_stream_backward_keeps_its_workspace():
    import torch
    q, k, v = _inputs(1, 16, 4096, 128, torch.float16, 5)
    o, lse = fa.attention_forward(q, k, v)
    do = torch.randn_like(q)
    ref = fa.attention_backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    ws_floats = fa.fa_bwd_workspace_size(1, 16, 4096, 128) // 4
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    got = fa.attention_backward(q, k, v, o, lse, do, stream=s)
    # the default stream at once asks for blocks of the workspace's size and
    # writes them while the side stream's kernels may still be running
    junk = [torch.full((ws_floats,), float("nan"), device="cuda:0") for _ in range(4)]
    torch.cuda.synchronize()
    assert _same(got, ref)
    assert all(bool(torch.isnan(j).all()) for j in junk)
    assert fa.fa_check(0) == fa.FA_OK


_THREADS_SCRIPT = r"""
import sys, threading
import torch
sys.path.insert(0, sys.argv[1])
import attention_forward_flashattention_gb300 as fa
fa.load_library()
torch.cuda.init()
# 8 host threads make their first calls at the same moment (the per-device
# setup of every entry point runs under its lock), each on a stream of its own
shapes = [(1, 4, 300 + 97 * i, 64 if i % 2 else 128, torch.float16 if i % 3 else torch.bfloat16,
           bool(i % 2)) for i in range(8)]
ins = []
for i, (B, H, N, d, dt, c) in enumerate(shapes):
    g = torch.Generator(device="cuda:0").manual_seed(100 + i)
    ins.append([torch.randn(B, H, N, d, device="cuda:0", generator=g).to(dt) for _ in range(3)])
torch.cuda.synchronize()
start = threading.Barrier(8)
got, errs = [None] * 8, []
def work(i):
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.default_stream())
        start.wait()
        for _ in range(4):
            o, lse = fa.attention_forward(*ins[i], causal=shapes[i][5], stream=s)
        s.synchronize()
        got[i] = (o, lse)
    except Exception as e:  # reported below
        errs.append(repr(e))
ts = [threading.Thread(target=work, args=(i,)) for i in range(8)]
[t.start() for t in ts]
[t.join() for t in ts]
assert not errs, errs
for i in range(8):
    o, lse = fa.attention_forward(*ins[i], causal=shapes[i][5])
    torch.cuda.synchronize()
    assert torch.equal(o, got[i][0]) and torch.equal(lse, got[i][1]), i
assert fa.fa_check(0) == fa.FA_OK
print("threads ok")
"""


def test_first_calls_from_many_host_threads():
    """A fresh process whose first calls come from 8 host threads at once,
    each on its own stream: no error, and every result equals the same call
    made afterwards alone."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _THREADS_SCRIPT, root], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout + r.stderr
