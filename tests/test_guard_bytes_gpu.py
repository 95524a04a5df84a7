"""Guard-byte (canary) checks of every buffer the library writes.

compute-sanitizer is not available on the GPUs these tests run on, so
out-of-bounds writes are caught the old way: every output, workspace and
cache buffer is carved out of a larger allocation whose 4 KiB on either side
hold a known byte pattern, and after the call (and a synchronize) both guard
regions must still hold it.  Covered: the tensor-core scoring path (W*g = 128
and 256), the CUDA-core path (fp32), per-query-head selection (its scores are
added into the zeroed score array), the LSE-input and all-query variants,
keep-all sequences, a 380 000-token prompt, the score-only entry point, the
host-buffer entry point's staging buffer, the entry point without a
workspace, both decode cache layouts and the Scissorhands cache across an
eviction.  The computed values themselves are checked elsewhere
(tests/parity.py and the other GPU tests); here a call must also leave its
indices valid.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from prefill_kv_cache_gb300 import scissorhands as SH
from prefill_kv_cache_gb300 import snapkv as S
from synth.device import make_layer_device
from tests import parity

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of pattern on each side (keeps 256-byte alignment)


def _pattern(n: int, salt: int) -> torch.Tensor:
    i = np.arange(n, dtype=np.int64)
    return torch.from_numpy(((i * 131 + 7 * salt + 29) % 251).astype(np.uint8))


class Guarded:
    """Device (or pinned host) allocations with patterned guard bytes."""

    def __init__(self, device="cuda", pinned=False):
        self.device, self.pinned, self.bufs = device, pinned, []

    def empty(self, shape, dtype, name):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        pat = _pattern(2 * GUARD + n, len(self.bufs) + 1)
        if self.pinned:
            buf = pat.clone().pin_memory()
        else:
            buf = pat.to(self.device)
        self.bufs.append((name, buf, pat))
        return buf[GUARD:GUARD + n].view(dtype).view(shape)

    def check(self):
        torch.cuda.synchronize()
        for name, buf, pat in self.bufs:
            host = buf.cpu()
            for side, sl in (("before", slice(0, GUARD)), ("after", slice(-GUARD, None))):
                bad = torch.nonzero(host[sl] != pat[sl]).flatten()
                assert bad.numel() == 0, f"{name}: {bad.numel()} guard bytes {side} overwritten"


def _outputs(G, B, C, H_out, d, dtype):
    return (G.empty((B, C, H_out, d), dtype, "out_k"), G.empty((B, C, H_out, d), dtype, "out_v"),
            G.empty((B, H_out, C), torch.int32, "out_idx"))


def _assert_indices(oi, seqlens, W, C):
    idx = oi.cpu().numpy()
    n = C - W
    for b, L in enumerate(seqlens):
        for row in idx[b]:
            if L > C:
                assert row[n:].tolist() == list(range(L - W, L))
                assert (np.diff(row[:n]) > 0).all() and row[:n].min(initial=0) >= 0
                assert row[:n].max(initial=0) < L - W
            else:
                assert row.tolist() == list(range(L)) + [-1] * (C - L)


def _compress_guarded(lay_or_dev, seqlens, H_q, H_kv, d, W, C, kp, pool, flags=0, lse=None):
    q, k, v = lay_or_dev
    B = len(seqlens)
    G = Guarded()
    H_out = H_q if flags & S.PER_QUERY_HEAD else H_kv
    ok, ov, oi = _outputs(G, B, C, H_out, d, k.dtype)
    shape = S.make_shape(B, H_q, H_kv, d, k.dtype)
    ws = G.empty((S.workspace_size(shape, seqlens, W, C, flags),), torch.uint8, "workspace")
    S.compress(q, k, v, seqlens, W, kp, pool, C, out_k=ok, out_v=ov, out_idx=oi, workspace=ws,
               flags=flags, lse_win=lse)
    assert S.get_status(ws) == S.OK
    G.check()
    _assert_indices(oi, seqlens, W, C)
    return ok, ov, oi, ws


CASES = [
    # seqlens,                 H_q, H_kv, d,  W,  C,   k, pool,  dtype, flags  (path)
    ([6000, 700, 3100],         32,   8, 128, 64, 1024, 13, "avg", "bf16", 0),  # tcgen05, 256 rows
    ([5000, 1100, 40],          32,   8, 128, 32, 1024, 7, "max", "bf16", 0),   # tcgen05, 128 rows
    ([2049, 130],               16,   4, 64, 32, 512,  5, "avg", "bf16", 0),    # tcgen05, d = 64
    ([4097, 300],               16,   2, 128, 16, 512, 3, "max", "fp32", 0),    # CUDA cores
    ([1025, 300, 2000],          8,   2, 128, 16, 256, 7, "max", "bf16", 0),    # CUDA cores (W*g = 64)
    ([5000, 600],               32,   8, 128, 32, 1024, 7, "avg", "bf16", 1),   # per query head
    ([3000, 900],                8,   8, 64, 16, 256,  5, "avg", "fp32", 1),    # per query head, g = 1
    ([33, 17, 1],                4,   2, 64, 16, 40,   5, "avg", "bf16", 0),    # all keep-all
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"L{c[0]}-g{c[1]//c[2]}-d{c[3]}-W{c[4]}-{c[8]}-f{c[9]}")
def test_compress_guards(case):
    seqlens, H_q, H_kv, d, W, C, kp, pool, dtype, flags = case
    lay = synth.make_inputs(401 + sum(seqlens), seqlens, H_q, H_kv, d, W, dtype, nspans=3)
    dev = tuple(parity.to_device(x) for x in (lay.q_win, lay.k, lay.v))
    _compress_guarded(dev, seqlens, H_q, H_kv, d, W, C, kp, pool, flags=flags)


def test_compress_with_lse_guards():
    seqlens, C = [5000, 800, 2500], 1024
    lay = synth.make_inputs(411, seqlens, 32, 8, 128, 32, "bf16", nspans=3)
    lse = parity.to_device(parity.window_lse(lay, C))
    dev = tuple(parity.to_device(x) for x in (lay.q_win, lay.k, lay.v))
    _compress_guarded(dev, seqlens, 32, 8, 128, 32, C, 5, "avg", lse=lse)


def test_prompt_380k_guards():
    q, k, v, seqlens = make_layer_device("5b", 0)
    cfg = synth.CONFIGS["5b"]
    _compress_guarded((q, k, v), seqlens, cfg["H_q"], cfg["H_kv"], cfg["d"], cfg["W"], cfg["C"],
                      cfg["k_pool"], cfg["pool"])


def test_score_only_guards():
    seqlens, W, C = [7000, 300], 64, 1024
    lay = synth.make_inputs(421, seqlens, 32, 8, 128, W, "bf16", nspans=3)
    q, k = parity.to_device(lay.q_win), parity.to_device(lay.k)
    shape = S.make_shape(2, 32, 8, 128, q.dtype)
    G = Guarded()
    ws = G.empty((S.workspace_size(shape, seqlens, W, C),), torch.uint8, "workspace")
    S.score(q, k, seqlens, W, C, ws)
    assert S.get_status(ws) == S.OK
    G.check()


def test_all_queries_guards():
    seqlens, W, C, H_q, H_kv, d = [1500, 200], 16, 256, 8, 2, 64
    lay = synth.make_inputs(431, seqlens, H_q, H_kv, d, W, "bf16", nspans=2)
    k, v = parity.to_device(lay.k), parity.to_device(lay.v)
    T = sum(seqlens)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(3)
    q_all = torch.randn((T, H_q, d), generator=gen, device="cuda").to(torch.bfloat16)
    lse_all = torch.full((T, H_q), 30.0, dtype=torch.float32, device="cuda")
    G = Guarded()
    ok, ov, oi = _outputs(G, 2, C, H_kv, d, torch.bfloat16)
    shape = S.make_shape(2, H_q, H_kv, d, torch.bfloat16)
    ws = G.empty((S.workspace_size(shape, seqlens, W, C),), torch.uint8, "workspace")
    arr, _ = S._seqlens_array(seqlens)
    rc = S.load().snapkv_compress_all_queries(
        ctypes.byref(shape), q_all.data_ptr(), k.data_ptr(), v.data_ptr(), lse_all.data_ptr(),
        arr, W, 5, S.POOL_AVG, C, ok.data_ptr(), ov.data_ptr(), oi.data_ptr(), ws.data_ptr(),
        ws.numel(), None)
    assert rc == S.OK
    G.check()
    _assert_indices(oi, seqlens, W, C)


def test_noalloc_guards():
    seqlens, W, C = [6000, 500], 32, 1024
    lay = synth.make_inputs(441, seqlens, 32, 8, 128, W, "bf16", nspans=3)
    q, k, v = (parity.to_device(x) for x in (lay.q_win, lay.k, lay.v))
    G = Guarded()
    ok, ov, oi = _outputs(G, 2, C, 8, 128, torch.bfloat16)
    S.compress_noalloc(q, k, v, seqlens, W, 7, "max", C, ok, ov, oi)
    G.check()
    _assert_indices(oi, seqlens, W, C)


def test_host_entry_point_guards():
    seqlens, W, C = [4000, 700], 32, 1024
    lay = synth.make_inputs(451, seqlens, 32, 8, 128, W, "bf16", nspans=3)
    q, k, v = (torch.from_numpy(x).view(torch.bfloat16).pin_memory()
               for x in (lay.q_win, lay.k, lay.v))
    H = Guarded(pinned=True)
    ok, ov, oi = _outputs(H, 2, C, 8, 128, torch.bfloat16)
    shape = S.make_shape(2, 32, 8, 128, S.BF16)
    D = Guarded()
    staging = D.empty((S.host_staging_size(shape, seqlens, W, C),), torch.uint8, "staging")
    S.compress_host(q, k, v, seqlens, W, 7, "avg", C, ok, ov, oi, staging)
    H.check()
    D.check()
    _assert_indices(oi, seqlens, W, C)


@pytest.mark.parametrize("layout", [S.CACHE_PACKED, S.CACHE_SLOTS])
def test_decode_guards(layout):
    B, H_q, H_kv, d, C = 3, 32, 8, 128, 1024
    lens = [131072, 1000, 5] if layout == S.CACHE_PACKED else [1024, 1000, 5]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    rows = sum(lens) if layout == S.CACHE_PACKED else B * C
    shp = (rows, H_kv, d) if layout == S.CACHE_PACKED else (B, C, H_kv, d)
    k = torch.randn(shp, generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn(shp, generator=gen, device="cuda").to(torch.bfloat16)
    q = torch.randn((B, H_q, d), generator=gen, device="cuda").to(torch.bfloat16)
    shape = S.make_shape(B, H_q, H_kv, d, torch.bfloat16)
    G = Guarded()
    out = G.empty((B, H_q, d), torch.float32, "out")
    ws = G.empty((S.decode_workspace_size(shape, lens, layout, C),), torch.uint8, "workspace")
    S.decode_attention(q, k, v, lens, layout, C, out=out, workspace=ws)
    G.check()
    assert torch.isfinite(out).all()


def test_scissorhands_guards():
    B, H_q, H_kv, d = 2, 16, 4, 128
    prm = SH.Params(budget=256, recent=8, history=40, evict=128)
    shape = S.make_shape(B, H_q, H_kv, d, torch.bfloat16)
    G = Guarded()
    cap, hw = prm.budget + 1, (prm.history + 31) // 32
    bufs = [G.empty((B, cap, H_kv, d), torch.bfloat16, "k"),
            G.empty((B, cap, H_kv, d), torch.bfloat16, "v"),
            G.empty((B, H_kv, cap), torch.int32, "pos"),
            G.empty((B, H_kv, hw, cap), torch.int32, "hist"),
            G.empty((B, 4), torch.int32, "state")]
    for t, w in zip(bufs, range(5)):
        assert t.numel() * t.element_size() == SH.buffer_bytes(shape, prm, w)
    ws = G.empty((SH.workspace_size(shape, prm),), torch.uint8, "workspace")
    out = G.empty((B, H_q, d), torch.float32, "out")
    c = SH.Cache.__new__(SH.Cache)
    c.shape, c.params, c.dtype = shape, prm, torch.bfloat16
    c.k, c.v, c.pos, c.hist, c.state = bufs
    c.workspace = ws
    c._c = SH.scissorhands_cache(*(t.data_ptr() for t in bufs))
    c._p = prm.c()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(9)
    rnd = lambda *s: torch.randn(s, generator=gen, device="cuda").to(torch.bfloat16)
    c.init([256, 100], [5000, 100], rnd(B, 256, H_kv, d), rnd(B, 256, H_kv, d))
    for _ in range(200):  # the first sequence starts full: evictions from step 1 on
        c.step(rnd(B, H_q, d), rnd(B, H_kv, d), rnd(B, H_kv, d), out=out)
    G.check()
    st = c.state.cpu().numpy()
    assert (st[:, 0] <= prm.budget).all() and (st[:, 0] >= 1).all()
