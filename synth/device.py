"""The hot-span generator drawn on the GPU, for benchmark-sized workloads.

Same recipe as ``synth.workloads`` (K, V ~ N(0,1) rounded to bf16; hot spans
of 8 prefix positions per KV head; window query = 2 * k[pos] + N(0,1)), drawn
with torch's seeded device generator so that 32 layers of 128K tokens take
milliseconds instead of minutes.  The arrays differ from the numpy draw (a
different random stream) but have the same shapes, distributions and
structure.  Like the rest of ``synth`` it holds none of the method's
arithmetic.
"""
from __future__ import annotations

import torch

from .workloads import CONFIGS, SPAN_LEN, config_seqlens


def make_layer_device(name: str, layer: int = 0, device: str = "cuda"):
    """(q_win [B,W,H_q,d], k [T,H_kv,d], v, seqlens list) on `device`."""
    cfg = CONFIGS[name]
    seqlens = config_seqlens(name)
    H_q, H_kv, d, W = cfg["H_q"], cfg["H_kv"], cfg["d"], cfg["W"]
    g = H_q // H_kv
    dt = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
    gen = torch.Generator(device=device)
    gen.manual_seed(1_000_003 * (cfg["seed_base"] + layer) + 17)
    T = sum(seqlens)
    k = torch.randn((T, H_kv, d), generator=gen, device=device, dtype=torch.float32).to(dt)
    v = torch.randn((T, H_kv, d), generator=gen, device=device, dtype=torch.float32).to(dt)
    qs = []
    off = 0
    for L in seqlens:
        P = L - W
        noise = torch.randn((W, H_q, d), generator=gen, device=device, dtype=torch.float32)
        ns = cfg["nspans"](L) if callable(cfg["nspans"]) else cfg["nspans"]
        if P >= 1 and ns >= 1:
            span = min(SPAN_LEN, P)
            starts = torch.randint(0, P - span + 1, (H_kv, ns), generator=gen, device=device)
            pick = torch.randint(0, ns, (W, H_q), generator=gen, device=device)
            within = torch.randint(0, span, (W, H_q), generator=gen, device=device)
            kvh = torch.arange(H_q, device=device) // g                   # [H_q]
            pos = starts[kvh.expand(W, H_q), pick] + within                # [W, H_q]
            rows = k[off + pos, kvh.expand(W, H_q)].float()                # [W, H_q, d]
            q = 2.0 * rows + noise
        else:
            q = noise
        qs.append(q.to(dt))
        off += L
    return torch.stack(qs).contiguous(), k, v, seqlens
