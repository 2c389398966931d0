"""ubatch_attention_static_scratch (attention with its split-K scratch in a
fixed device array, no memory obtained during the call) against
ubatch_attention, through the C interface.

Collected last on purpose: it must pass alone and after every other test has
used the device (the scratch array is shared by all calls on a device).
"""

import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

from workloads import configs
from tests.gpu_util import Pair, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import continuous_batching_kv_gb300  # noqa: F401  (fails loudly if the library is missing)


def _prepared(p, call):
    """Split, reserve and store every layer of `call`; returns the split handle
    and, per ubatch, its rows' q as device tensors per layer."""
    kv, torch = p.kv, p.torch
    s = kv.kv_split_ubatches(p.c, call["pos"], call["seq"])
    assert kv.kv_prepare_cells(p.c, s) == 0
    qs = []
    for k in range(kv.kv_split_count(s)):
        rows = list(kv.kv_split_ubatch(s, k)["rows"])
        pos = [call["pos"][r] for r in rows]
        con = [call["content"][r] for r in rows]
        ql = []
        for layer in range(p.L):
            q, kk, vv = p.qkv(layer, pos, con)
            kv.kv_store(p.c, s, k, layer, torch.from_numpy(kk).cuda(), torch.from_numpy(vv).cuda())
            ql.append(torch.from_numpy(q).cuda())
        qs.append(ql)
    return s, qs


def _attend(p, fn, s, k, layer, q):
    n = q.shape[0]
    o = p.torch.full((n, p.H, p.d), float("nan"), dtype=p.torch.float32, device="cuda")
    fn(p.c, s, k, layer, q, o)
    p.torch.cuda.synchronize()
    assert p.kv.kv_device_error(p.c) == 0
    return o.cpu().numpy()


def test_static_scratch_matches_ubatch_attention_two_calls():
    # eight sequences with contexts 64 .. 2048, one decode row each, two layers
    cfg = configs.config(3, n_layer=2)
    p = Pair(cfg, oracle=False)
    kv = p.kv
    try:
        for call in cfg["setup"]:
            s, _ = _prepared(p, call)
            kv.kv_split_free(s)
        s, qs = _prepared(p, cfg["measured"][0])
        assert kv.kv_split_count(s) == 1
        for layer in (0, 1, 1):   # two calls in a row on different layers, then a repeat
            q = qs[0][layer]
            ref = _attend(p, kv.ubatch_attention, s, 0, layer, q)
            got = _attend(p, kv.ubatch_attention_static_scratch, s, 0, layer, q)
            check_close(got, ref.astype(np.float64), "layer %d" % layer)
        kv.kv_split_free(s)
    finally:
        p.close()


def test_static_scratch_rejects_prefill_and_oversize():
    import torch
    kv = pytest.importorskip("continuous_batching_kv_gb300")
    # a 100-token prompt: its block takes the tensor-core prefill path
    cfg = {"id": 11, "name": "static-prefill", "shape": dict(configs.QWEN, n_layer=1),
           "params": dict(n_ctx=256, n_batch=256, n_ubatch=128, n_seq_max=1, n_stream=1),
           "setup": [], "measured": []}
    p = Pair(cfg, oracle=False)
    try:
        s, qs = _prepared(p, {"pos": list(range(100)), "seq": [[0]] * 100, "content": [0] * 100})
        o = torch.zeros((100, p.H, p.d), dtype=torch.float32, device="cuda")
        with pytest.raises(kv.KvError) as e:
            kv.ubatch_attention_static_scratch(p.c, s, 0, 0, qs[0][0], o)
        assert e.value.code == kv.KV_E_INVAL
        kv.kv_split_free(s)
    finally:
        p.close()
    # 256 one-row sequences with 16 KV heads: more split-K scratch than the array holds
    n = 256
    cfg = {"id": 12, "name": "static-oversize",
           "shape": dict(n_head=32, n_head_kv=16, head_dim=128, n_layer=1),
           "params": dict(n_ctx=n, n_batch=n, n_ubatch=n, n_seq_max=n, n_stream=1),
           "setup": [], "measured": []}
    p = Pair(cfg, oracle=False)
    try:
        s, qs = _prepared(p, {"pos": [0] * n, "seq": [[i] for i in range(n)], "content": [0] * n})
        o = torch.zeros((n, p.H, p.d), dtype=torch.float32, device="cuda")
        with pytest.raises(kv.KvError) as e:
            kv.ubatch_attention_static_scratch(p.c, s, 0, 0, qs[0][0], o)
        assert e.value.code == kv.KV_E_INVAL
        assert "scratch" in str(e.value)
        # the regular entry point still serves it
        kv.ubatch_attention(p.c, s, 0, 0, qs[0][0], o)
        torch.cuda.synchronize()
        assert kv.kv_device_error(p.c) == 0
        kv.kv_split_free(s)
    finally:
        p.close()


# Run in a fresh process: nothing of the library has touched the device before
# kv_init, so a module load or an allocation made by the first static-scratch
# call would show as a drop in the device's free memory.
_FRESH = textwrap.dedent("""
    import sys, torch
    sys.path.insert(0, {root!r})
    import continuous_batching_kv_gb300 as kv
    from workloads import configs
    from tests.gpu_util import Pair
    from tests.test_zz_no_alloc import _prepared
    cfg = configs.config(3, n_layer=1)
    p = Pair(cfg, oracle=False)
    for call in cfg["setup"]:
        s, _ = _prepared(p, call)
        kv.kv_split_free(s)
    s, qs = _prepared(p, cfg["measured"][0])
    q = qs[0][0]
    o = torch.empty((q.shape[0], p.H, p.d), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    lib0 = kv.kv_device_bytes(p.c)
    kv.ubatch_attention_static_scratch(p.c, s, 0, 0, q, o)
    torch.cuda.synchronize()
    assert kv.kv_device_error(p.c) == 0
    free1 = torch.cuda.mem_get_info()[0]
    lib1 = kv.kv_device_bytes(p.c)
    kv.ubatch_attention_static_scratch(p.c, s, 0, 0, q, o)
    torch.cuda.synchronize()
    free2 = torch.cuda.mem_get_info()[0]
    print("FREE", free0, free1, free2, "LIB", lib0, lib1)
    assert free0 == free1 == free2, (free0, free1, free2)
    assert lib0 == lib1, (lib0, lib1)
    kv.kv_split_free(s)
    p.close()
""")


def test_static_scratch_first_call_obtains_no_memory():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH.format(root=root)], cwd=root,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "FREE" in r.stdout
