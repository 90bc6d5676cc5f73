"""Seeded synthetic workloads for the compressed-KV decode path.

This module only draws inputs: it holds none of the method's arithmetic (no
quantiser, no score, no selection, no attention).  Both the CUDA path and the
CPU oracle are fed from it.

Recipe (the same for every vector: queries, indexer queries, cache entries,
window rows): draw N(0, 1) per channel, divide by the vector's RMS (no gain),
round to BF16.  This stands in for the post-RMSNorm latents the pages
describe ("V4.1-Flash 공개", 핵심 내용: the RMSNorm output stays near 22.6 at
most, i.e. sqrt(512) for a 512-d vector of unit RMS).  Head weights of the
indexer are U(0, 1).  The optional spike recipe replaces one entry in 64, before
normalisation, by A * e_m + 0.01 * N(0, 1) (random channel m, A = 100), so that
its largest coordinate approaches sqrt(512) after normalisation.  The optional
tie recipe copies the vectors of donor entries onto 5 % of the other entries
(see ``inject_ties``).

Random streams are torch Philox/MT generators seeded per tensor and per
sequence from the workload seed, so a subset of sequences can be regenerated
alone on the host for the oracle.
"""

from dataclasses import dataclass, field
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str              # 'csa', 'hca' or 'csa2'
    B: int
    T: int                 # context tokens
    ratio: int             # 4 (CSA) or 128 (HCA)
    H: int                 # query heads
    HI: int                # indexer heads (0 for HCA)
    topk: int
    W: int                 # sliding window
    main_fmt: str          # 'bf16' | 'mixed' | 'fp4'
    idx_fmt: str           # 'bf16' | 'fp4' | ''
    seed: int
    ties: bool = False
    spikes: bool = False
    pool_len: int = 0
    n_append: int = 0
    n_layers: int = 1
    nope_block: int = 448  # channels per f32 scale of the MIXED format
    D: int = 512
    R: int = 64
    DI: int = 128

    @property
    def n_comp(self) -> int:
        return self.T // self.ratio

    @property
    def tau(self) -> float:
        return 1.0 / math.sqrt(self.D)


WORKLOADS = {
    # Tiny CSA decode, BF16 everywhere.
    "csa_tiny_4k": Workload("csa_tiny_4k", "csa", B=1, T=4096, ratio=4, H=16, HI=4, topk=512,
                            W=128, main_fmt="bf16", idx_fmt="bf16", seed=1000),
    # CSA decode at V4-Pro layer shapes, 128k context, mixed storage.
    "csa_128k": Workload("csa_128k", "csa", B=8, T=131072, ratio=4, H=128, HI=64, topk=512,
                         W=128, main_fmt="mixed", idx_fmt="fp4", seed=1001),
    # HCA decode, dense over 1M/128 BF16 entries.
    "hca_1m": Workload("hca_1m", "hca", B=16, T=1048576, ratio=128, H=128, HI=0, topk=0,
                       W=128, main_fmt="bf16", idx_fmt="", seed=1002),
    # CSA decode at V4-Pro's own indexer setting: top-1024, and FP8 scales per
    # 64 channels (the act_quant block reading), 128k context.
    "csa_128k_pro": Workload("csa_128k_pro", "csa", B=8, T=131072, ratio=4, H=128, HI=64, topk=1024,
                             W=128, main_fmt="mixed", idx_fmt="fp4", seed=1005, nope_block=64),
    # CSA decode at 1M context with ~5 % exact score ties.
    "csa_1m": Workload("csa_1m", "csa", B=4, T=1048576, ratio=4, H=128, HI=64, topk=512,
                       W=128, main_fmt="mixed", idx_fmt="fp4", seed=1003, ties=True),
    # CSA2 six-layer group, FP4 main KV, 256k context, 64 appended rows.
    "csa2_group": Workload("csa2_group", "csa2", B=8, T=262144, ratio=4, H=64, HI=64, topk=512,
                           W=128, main_fmt="fp4", idx_fmt="fp4", seed=1004, spikes=True,
                           pool_len=2048, n_append=64, n_layers=6),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def _stream_seed(seed: int, tag: int, b: int = 0) -> int:
    return seed * 1_000_003 + tag * 10_007 + b


def rms_rows(shape, seed: int, device="cpu", spikes: bool = False,
             spike_every: int = 64, spike_amp: float = 100.0) -> torch.Tensor:
    """BF16 tensor of RMS-normalised N(0,1) vectors along the last axis."""
    g = _gen(device, seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if spikes and x.numel():
        rows = x.reshape(-1, shape[-1])
        n = rows.shape[0]
        pick = torch.rand(n, generator=g, device=device) < (1.0 / spike_every)
        chan = torch.randint(0, shape[-1], (n,), generator=g, device=device)
        noise = 0.01 * torch.randn(rows.shape, generator=g, device=device)
        spike = noise.clone()
        spike[torch.arange(n, device=device), chan] += spike_amp
        rows = torch.where(pick[:, None], spike, rows)
        x = rows.reshape(shape)
    rms = torch.sqrt(torch.mean(x * x, dim=-1, keepdim=True)).clamp_min(1e-30)
    return (x / rms).to(torch.bfloat16)


def head_weights(shape, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(device, seed)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


TAG_Q, TAG_QIDX, TAG_W, TAG_KV, TAG_IDXKEY, TAG_WIN, TAG_APPEND = range(7)


def sequence_rows(wl: Workload, b: int, n_comp: int, device="cpu", layer: int = 0):
    """Float inputs of sequence ``b`` (one layer): cache entries [n_comp, D],
    indexer keys [n_comp, DI] (CSA only) and window rows [W, D]."""
    sd = wl.seed + 7 * layer
    kv = rms_rows((n_comp, wl.D), _stream_seed(sd, TAG_KV, b), device, spikes=wl.spikes)
    win = rms_rows((wl.W, wl.D), _stream_seed(sd, TAG_WIN, b), device, spikes=wl.spikes)
    keys = None
    if wl.kind != "hca":
        keys = rms_rows((n_comp, wl.DI), _stream_seed(sd, TAG_IDXKEY, b), device)
    return kv, keys, win


def step_queries(wl: Workload, step: int = 0, device="cpu", layer: int = 0, batch=None):
    """Per-step inputs: q [B, H, D], q_idx [B, HI, DI], w [B, HI]."""
    bs = range(wl.B) if batch is None else batch
    sd = wl.seed + 7 * layer + 131 * step
    q = torch.stack([rms_rows((wl.H, wl.D), _stream_seed(sd, TAG_Q, b), device) for b in bs])
    if wl.HI:
        qi = torch.stack([rms_rows((wl.HI, wl.DI), _stream_seed(sd, TAG_QIDX, b), device)
                          for b in bs])
        w = torch.stack([head_weights((wl.HI,), _stream_seed(sd, TAG_W, b), device) for b in bs])
    else:
        qi, w = None, None
    return q, qi, w


def append_rows(wl: Workload, n: int, dim: int, step: int = 0, device="cpu") -> torch.Tensor:
    return rms_rows((n, dim), _stream_seed(wl.seed + 131 * step, TAG_APPEND), device,
                    spikes=wl.spikes)


def inject_ties(keys: torch.Tensor, ranking, seed: int, frac: float = 0.05,
                donor_lo: int = 480, donor_hi: int = 544) -> torch.Tensor:
    """Copy donor vectors onto ~``frac`` of the other entries.

    ``ranking`` lists the entry indices of one sequence from best to worst
    score (supplied by the caller); the donors are those ranked
    [donor_lo, donor_hi).  Recipients are drawn uniformly without replacement
    from the non-donors, each with a uniformly drawn donor.  Identical
    vectors quantise to identical bytes, so every recipient ties exactly with
    its donor, and the copies crowd the top-k boundary.
    """
    n = keys.shape[0]
    ranking = torch.as_tensor(ranking, dtype=torch.int64).cpu()
    donors = ranking[donor_lo:donor_hi]
    mask = torch.ones(n, dtype=torch.bool)
    mask[donors] = False
    others = torch.nonzero(mask).flatten()
    g = _gen("cpu", seed)
    n_rec = int(round(frac * n))
    perm = torch.randperm(len(others), generator=g)[:n_rec]
    rec = others[perm]
    pick = donors[torch.randint(0, len(donors), (n_rec,), generator=g)]
    out = keys.clone()
    out[rec.to(keys.device)] = keys[pick.to(keys.device)]
    return out
