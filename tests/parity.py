"""GPU-vs-oracle agreement rule, shared by the GPU parity tests.

Rule (scores fp32 on the GPU, fp64 in the oracle):
  * pooled (and raw) scores: |gpu - oracle| <= 1e-7 + 1e-5 * |oracle|;
  * with tau the oracle's (C-W)-th best pooled score, the exemption set is
    E = {j : |pooled_oracle[j] - tau| <= 1e-5 * tau}; the kept prefix sets of
    GPU and oracle may differ only inside E (the count is reported);
  * every GPU output slot holds the exact bytes of the K and V rows of its
    own index (compared by index, since an exempt swap shifts later slots);
    unused slots (index -1) are zero; the kept prefix indices ascend; the
    window block is identical to the oracle's.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import synth
from prefill_kv_cache_gb300 import snapkv as S

RTOL = 1e-5
ATOL = 1e-7

# One record per check() call: the test that made it, the (sequence, head)
# units compared, the size of the exemption band E summed over them and the
# number of positions kept by exactly one side (all inside E).  conftest.py
# prints the table at the end of the session.
NEAR_TIES: list[dict] = []


def to_device(a: np.ndarray, dev="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(dev)


def window_lse(lay, C, fill=np.nan):
    """Natural-log LSE of every window query row over its visible keys.

    fp64 on the CPU from the layer's (bf16-exact) inputs, returned as fp32
    [B, W, H_q], the input of snapkv_compress_with_lse: row (b, i, head) is
    log sum_{j <= L_b - W + i} exp(q . k_j / sqrt(d)) with k from the head's
    KV group.  Sequences with L_b <= C are filled with `fill` (the library
    must not read them).
    """
    B, W, H_q, d = lay.q_win.shape
    g = H_q // lay.H_kv
    out = np.full((B, W, H_q), fill, dtype=np.float32)
    q_all = lay.q_win if lay.q_win.dtype != np.uint16 else synth.bf16_to_f32(lay.q_win)
    k_all = lay.k if lay.k.dtype != np.uint16 else synth.bf16_to_f32(lay.k)
    for b, L in enumerate(lay.seqlens):
        L = int(L)
        if L <= C:
            continue
        P = L - W
        kb = torch.from_numpy(np.ascontiguousarray(k_all[lay.offsets[b]:lay.offsets[b] + L]))
        kb = kb.to(torch.float64)
        mask = torch.arange(L)[None, :] > (P + torch.arange(W))[:, None]  # [W, L]
        for h in range(lay.H_kv):
            q = torch.from_numpy(np.ascontiguousarray(q_all[b, :, h * g:(h + 1) * g]))
            s = torch.einsum("imd,jd->mij", q.to(torch.float64), kb[:, h]) / np.sqrt(d)
            s.masked_fill_(mask[None], -np.inf)
            out[b, :, h * g:(h + 1) * g] = torch.logsumexp(s, dim=2).T.numpy()
    return out


def run_gpu(lay, k_pool, pool, C, dev="cuda", lse=None, flags=0):
    """One snapkv_compress (snapkv_compress_with_lse when `lse` is given,
    snapkv_compress_ex when flags are) on the layer; returns numpy outputs
    and scores."""
    q = to_device(lay.q_win, dev)
    k = to_device(lay.k, dev)
    v = to_device(lay.v, dev)
    lse_t = None if lse is None else to_device(lse, dev)
    ok, ov, oi, ws = S.compress(q, k, v, lay.seqlens, lay.W, k_pool, pool, C, lse_win=lse_t,
                                flags=flags)
    st = S.get_status(ws)
    assert st == S.OK, S.status_string(st)
    shape = S.make_shape(lay.B, lay.H_q, lay.H_kv, lay.d, q.dtype)
    raw, pooled = S.scores_from_workspace(ws, shape, lay.seqlens, lay.W, C, flags)
    torch.cuda.synchronize()

    def host(t):
        t = t.cpu()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    return dict(out_k=host(ok), out_v=host(ov), idx=oi.cpu().numpy(), raw=raw.cpu().numpy(),
                pooled=pooled.cpu().numpy())


def unpack_scores(vec, seqlens, H_kv, W, C):
    """Split a packed (b, h, j) score vector into per-sequence [H_kv, P] arrays."""
    out, off = [], 0
    for L in seqlens:
        L = int(L)
        if L > C:
            P = L - W
            out.append(vec[off:off + H_kv * P].reshape(H_kv, P))
            off += H_kv * P
        else:
            out.append(None)
    return out


# The LSE-input entry points compare logits the GPU accumulates in fp32 on
# the tensor cores with an LSE computed exactly (fp64, then rounded to fp32)
# outside the library.  With the two-pass path the rounding of a row's
# dominant logit appears both in the row's LSE and in its own term and
# cancels; with an outside LSE it does not: a logit of ~22 nats (q . k ~ 256
# summed over d = 128 products in fp32) carries ~1e-5 of absolute rounding,
# i.e. ~1e-5 of relative error in its probability, on top of the fp32
# roundings of the LSE itself and of log2(e) / sqrt(d).  The LSE-input tests
# therefore use twice the two-pass tolerance, for the scores and the
# exemption band alike.
LSE_RTOL = 2e-5


def check(lay, gpu, ora, C, seqs=None, heads=None, report=None, rtol=RTOL):
    """Assert the agreement rule on sequences `seqs` (default all) of `lay`.

    `ora` holds the oracle's outputs for exactly those sequences, in order.
    Returns the number of exempt swaps seen.
    """
    W, H_kv = lay.W, lay.H_kv
    n = C - W
    seqs = list(range(lay.B)) if seqs is None else list(seqs)
    heads = list(range(H_kv)) if heads is None else list(heads)
    g_raw = unpack_scores(gpu["raw"], lay.seqlens, H_kv, W, C)
    g_pool = unpack_scores(gpu["pooled"], lay.seqlens, H_kv, W, C)
    offs = lay.offsets
    swaps = 0
    band = 0      # |E| summed over the scored units
    decided = 0   # positions in E kept by exactly one side
    units = 0
    for oi_, b in enumerate(seqs):
        L = int(lay.seqlens[b])
        P = L - W
        for h in heads:
            gi = gpu["idx"][b, h]
            oi = ora["idx"][oi_, h]
            tag = f"seq {b} head {h}"
            if L > C:
                np.testing.assert_allclose(g_raw[b][h], ora["raw"][oi_][h], rtol=rtol, atol=ATOL,
                                           err_msg=f"raw scores, {tag}")
                np.testing.assert_allclose(g_pool[b][h], ora["pooled"][oi_][h], rtol=rtol,
                                           atol=ATOL, err_msg=f"pooled scores, {tag}")
                assert gi[n:].tolist() == list(range(P, L)), f"window block, {tag}"
                sel_g = gi[:n]
                assert (np.diff(sel_g) > 0).all() and sel_g.min(initial=0) >= 0 and \
                    sel_g.max(initial=0) < P, f"kept indices not ascending in [0,P), {tag}"
                tau = ora["tau"][oi_, h]
                po = ora["pooled"][oi_][h]
                units += 1
                if n > 0:
                    band += int(np.count_nonzero(np.abs(po - tau) <= rtol * tau))
                diff = set(sel_g.tolist()) ^ set(oi[:n].tolist())
                if diff:
                    bad = [j for j in diff if abs(po[j] - tau) > rtol * tau]
                    assert not bad, f"kept sets differ outside the exemption band, {tag}: {bad[:8]}"
                    swaps += len(diff) // 2
                    decided += len(diff)
            else:
                assert gi.tolist() == oi.tolist(), f"keep-all indices, {tag}"
            # bytes by index
            rows = gi >= 0
            src = offs[b] + gi[rows]
            np.testing.assert_array_equal(gpu["out_k"][b, rows, h], lay.k[src, h], err_msg=tag)
            np.testing.assert_array_equal(gpu["out_v"][b, rows, h], lay.v[src, h], err_msg=tag)
            assert (gpu["out_k"][b, ~rows, h] == 0).all() and (gpu["out_v"][b, ~rows, h] == 0).all()
    if report is not None:
        report.append(swaps)
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    NEAR_TIES.append(dict(test=test, units=units, band=band, decided_in_band=decided,
                          swaps=swaps))
    return swaps


def oracle_for(lay, k_pool, pool, C, seqs=None, nthreads=None):
    """Oracle outputs on a subset of sequences (default all)."""
    if seqs is None:
        return oracle.compress(lay.q_win, lay.k, lay.v, lay.seqlens, lay.W, k_pool, pool, C,
                               nthreads=nthreads)
    seqs = list(seqs)
    offs = lay.offsets
    q = np.ascontiguousarray(lay.q_win[seqs])
    ks = np.concatenate([lay.k[offs[b]:offs[b] + lay.seqlens[b]] for b in seqs])
    vs = np.concatenate([lay.v[offs[b]:offs[b] + lay.seqlens[b]] for b in seqs])
    sl = [int(lay.seqlens[b]) for b in seqs]
    return oracle.compress(q, ks, vs, sl, lay.W, k_pool, pool, C, nthreads=nthreads)


def expand_heads(lay):
    """The layer with each KV head repeated for the g query heads it serves
    (H_kv := H_q): per-query-head selection on `lay` equals the plain
    compression of this layer."""
    import dataclasses
    g = lay.H_q // lay.H_kv
    return dataclasses.replace(lay, k=np.ascontiguousarray(np.repeat(lay.k, g, axis=1)),
                               v=np.ascontiguousarray(np.repeat(lay.v, g, axis=1)),
                               H_kv=lay.H_q,
                               targets=[[t[h // g] for h in range(lay.H_q)] for t in lay.targets])
