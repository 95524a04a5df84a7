"""Workload shapes and the hot-span input generator.

Shapes follow the workloads the SnapKV pages describe: a Llama-3-8B layer
(32 query heads, 8 KV heads, head dim 128) at 16K and 128K prompt tokens,
a Mistral-7B layer batch, a ragged batch and a single 380K-token prompt
("SnapKV: LLM Knows What You are Looking for Before Generation", abstract and
"주요 결과"; jisaku.com glossary "SnapKV", "性能評価").  Observation windows of
16-64 tokens, pooling kernels 5-13 and budgets of 1024-4096 come from the same
pages ("기술적 접근법").

Generator (the same for every workload):

* K and V ~ N(0, 1) in fp32, rounded to bf16 (round to nearest even) when the
  workload is bf16.
* Per (sequence, KV head): ``nspans`` hot spans of 8 consecutive prefix
  positions, start uniform in ``[0, P - 8]`` (P = L - W), overlaps allowed.
* Per (sequence, query head, window row): pick one span of the query head's
  KV group uniformly, then one position in it uniformly; the window query is
  ``2.0 * k[pos] + N(0, 1)`` (k already rounded), rounded like K.

All draws use numpy's PCG64 ``default_rng`` keyed by integer tuples, so the
arrays are identical on every machine.  Large tensors are drawn in fixed
4096-row chunks, each with its own key, so that chunks can be drawn on
several threads without changing the result.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

SPAN_LEN = 8
CHUNK_ROWS = 4096

# name -> workload description.  "nspans" is per KV head per sequence; a
# callable takes the sequence length.
CONFIGS: dict[str, dict] = {
    "1": dict(
        desc="tiny MHA layer: 4/4 heads, d=64, L=1024, fp32, W=16, avg k=5, C=256",
        H_q=4, H_kv=4, d=64, seqlens=[1024], dtype="fp32", W=16, k_pool=5,
        pool="avg", C=256, nspans=4, layers=1, seed_base=0,
    ),
    "2": dict(
        desc="Llama-3-8B layer, 16K prompt: 32/8 heads, d=128, bf16, W=32, max k=7, C=1024",
        H_q=32, H_kv=8, d=128, seqlens=[16384], dtype="bf16", W=32, k_pool=7,
        pool="max", C=1024, nspans=32, layers=1, seed_base=2000,
    ),
    "3": dict(
        desc="Mistral-7B layer, 8 x 32K prompts: 32/8 heads, d=128, bf16, W=32, avg k=5, C=2048",
        H_q=32, H_kv=8, d=128, seqlens=[32768] * 8, dtype="bf16", W=32,
        k_pool=5, pool="avg", C=2048, nspans=64, layers=1, seed_base=3000,
    ),
    "4": dict(
        desc="Llama-3-8B, 128K prompt, 32 layers: 32/8 heads, d=128, bf16, W=64, avg k=13, C=4096",
        H_q=32, H_kv=8, d=128, seqlens=[131072], dtype="bf16", W=64,
        k_pool=13, pool="avg", C=4096, nspans=128, layers=32, seed_base=4000,
    ),
    "5a": dict(
        desc="ragged batch of 16 prompts, L ~ U[4096, 65536]: 32/8 heads, d=128, bf16, W=32, max k=7, C=1024",
        H_q=32, H_kv=8, d=128, seqlens=None, dtype="bf16", W=32, k_pool=7,
        pool="max", C=1024, nspans=lambda L: L // 512, layers=1, seed_base=5000,
    ),
    "5b": dict(
        desc="one 380000-token prompt: 32/8 heads, d=128, bf16, W=32, max k=7, C=1024",
        H_q=32, H_kv=8, d=128, seqlens=[380000], dtype="bf16", W=32, k_pool=7,
        pool="max", C=1024, nspans=lambda L: L // 512, layers=1, seed_base=5500,
    ),
}


def config_seqlens(name: str) -> list[int]:
    cfg = CONFIGS[name]
    if cfg["seqlens"] is not None:
        return list(cfg["seqlens"])
    # ragged batch: 16 lengths uniform in [4096, 65536], seed 5000
    rng = np.random.default_rng(5000)
    return [int(x) for x in rng.integers(4096, 65537, 16)]


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (finite input)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32, exact."""
    return (np.ascontiguousarray(h).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Layer:
    """One layer's inputs in the packed layouts the library takes.

    q_win:   [B, W, H_q, d]  queries of the last W prompt positions
    k, v:    [T, H_kv, d]    packed varlen, T = sum(seqlens)
    seqlens: [B] int32
    Arrays are uint16 bf16 bit patterns when dtype == "bf16", else float32.
    targets[b][h] is the sorted set of prefix positions that some window
    query of KV group h was built from.
    """

    q_win: np.ndarray
    k: np.ndarray
    v: np.ndarray
    seqlens: np.ndarray
    dtype: str
    H_q: int
    H_kv: int
    d: int
    W: int
    targets: list

    @property
    def B(self) -> int:
        return len(self.seqlens)

    @property
    def offsets(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens)[:-1]]).astype(np.int64)


def _normal_rows(key: tuple, rows: int, row_shape: tuple, threads: int) -> np.ndarray:
    """N(0,1) fp32 array [rows, *row_shape] drawn in fixed 4096-row chunks."""
    out = np.empty((rows,) + tuple(row_shape), dtype=np.float32)
    nchunks = (rows + CHUNK_ROWS - 1) // CHUNK_ROWS

    def fill(c: int) -> None:
        r0 = c * CHUNK_ROWS
        r1 = min(rows, r0 + CHUNK_ROWS)
        rng = np.random.default_rng(list(key) + [c])
        out[r0:r1] = rng.standard_normal((r1 - r0,) + tuple(row_shape), dtype=np.float32)

    if threads > 1 and nchunks > 1:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fill, range(nchunks)))
    else:
        for c in range(nchunks):
            fill(c)
    return out


def _to_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_round(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def _make_seq(seed, b, L, H_q, H_kv, d, W, dtype, nspans, threads, q_scale=2.0):
    """Sequence b of a batch: (q [W,H_q,d], k [L,H_kv,d], v, targets per KV head)."""
    g = H_q // H_kv
    P = L - W
    kf = _normal_rows((seed, b, 0), L, (H_kv, d), threads)
    vf = _normal_rows((seed, b, 1), L, (H_kv, d), threads)
    kb = _to_dtype(kf, dtype)
    vb = _to_dtype(vf, dtype)
    kr = bf16_to_f32(kb) if dtype == "bf16" else kb
    ns = nspans(L) if callable(nspans) else int(nspans)
    rng = np.random.default_rng((seed, b, 2))
    noise = rng.standard_normal((W, H_q, d), dtype=np.float32)
    qf = noise.copy()
    sets = [set() for _ in range(H_kv)]
    if P >= 1 and ns >= 1:
        span = min(SPAN_LEN, P)
        starts = rng.integers(0, P - span + 1, (H_kv, ns))
        pick = rng.integers(0, ns, (W, H_q))
        within = rng.integers(0, span, (W, H_q))
        for i in range(W):
            for hq in range(H_q):
                h = hq // g
                pos = int(starts[h, pick[i, hq]] + within[i, hq])
                sets[h].add(pos)
                qf[i, hq] = np.float32(q_scale) * kr[pos, h] + noise[i, hq]
    return _to_dtype(qf, dtype), kb, vb, [sorted(s) for s in sets]


def make_inputs(
    seed: int,
    seqlens,
    H_q: int,
    H_kv: int,
    d: int,
    W: int,
    dtype: str = "bf16",
    nspans=4,
    threads: int | None = None,
    q_scale: float = 2.0,
    seq_ids=None,
) -> Layer:
    """Draw one layer with the hot-span generator (see module docstring).

    ``seq_ids`` gives each sequence's index within its batch (default
    0..B-1); a sequence's arrays depend only on (seed, its index, its length),
    so a sub-batch equals the matching slice of the full batch.
    """
    if H_q % H_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    if dtype not in ("bf16", "fp32"):
        raise ValueError(dtype)
    threads = threads or min(16, os.cpu_count() or 1)
    seqlens = np.asarray(list(seqlens), dtype=np.int32)
    seq_ids = list(range(len(seqlens))) if seq_ids is None else list(seq_ids)
    qs, ks, vs, targets = [], [], [], []
    for b, L in zip(seq_ids, seqlens):
        q, k, v, t = _make_seq(seed, b, int(L), H_q, H_kv, d, W, dtype, nspans,
                               threads, q_scale)
        qs.append(q)
        ks.append(k)
        vs.append(v)
        targets.append(t)
    return Layer(q_win=np.ascontiguousarray(np.stack(qs)),
                 k=np.ascontiguousarray(np.concatenate(ks)),
                 v=np.ascontiguousarray(np.concatenate(vs)),
                 seqlens=seqlens, dtype=dtype, H_q=H_q, H_kv=H_kv, d=d, W=W,
                 targets=targets)


def make_layer(name: str, layer: int = 0, seqs=None, threads: int | None = None) -> Layer:
    """Inputs of one layer of a named workload (``seqs``: a subset of its batch)."""
    cfg = CONFIGS[name]
    seqlens = config_seqlens(name)
    ids = list(range(len(seqlens))) if seqs is None else list(seqs)
    return make_inputs(cfg["seed_base"] + layer, [seqlens[b] for b in ids], cfg["H_q"],
                       cfg["H_kv"], cfg["d"], cfg["W"], cfg["dtype"], cfg["nspans"],
                       threads, seq_ids=ids)
