"""Seeded synthetic inputs for the routed-expert FP8 MoE FFN.

Shared by the tests, the benchmark and the smoke check.  This module draws
random numbers and routing decisions only: it holds none of the FFN's own
arithmetic (no FP8 quantisation, no GEMM, no SwiGLU, no combine), so the CPU
oracle and the CUDA library share nothing but the inputs they are handed.

Two generators are used:

* ``counter_normal`` / ``counter_uniform`` -- a counter-based generator written
  with integer torch ops only.  Value ``i`` of stream ``(seed, stream)`` is a
  pure function of ``i``, so the same tensor comes out on the CPU and on a GPU,
  and any slice (one expert, one 128-row block) can be regenerated alone.
  Large tensors (expert weights, activations) use it.  The normal variate is
  the Irwin-Hall sum of twelve 16-bit uniforms, centred and divided by 2^16:
  exact in float32, mean 0, variance 1 - 2^-32, support [-6, 6].
* numpy ``default_rng(1000 + config_index)`` -- small host-side draws: router
  logits, Zipf expert popularity, Gumbel top-k routing.

Workloads follow the DeepSeek-V3 MoE shapes the two SGLang deployment pages
run (hidden 7168, expert intermediate 2048, top-8 routing, a 288-expert pool
of 256 routed + 32 redundant experts for EPLB; "Deploying DeepSeek with PD
Disaggregation and Large-Scale Expert Parallelism on 96 H100 GPUs", section
"Expert Parallelism Load Balancer").
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = [
    "counter_normal", "counter_uniform", "bf16_normal", "MoEConfig", "CONFIGS",
    "get_config", "make_routing", "make_activations", "make_expert_weights",
    "zipf_split",
]

_M32 = 0xFFFFFFFF


# ----------------------------------------------------------------------------
# counter-based generator (device independent)
# ----------------------------------------------------------------------------
def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for int64 x in [0, 2^32) without int64 overflow."""
    return ((x & 0xFFFF) * c + (((x >> 16) * (c & 0xFFFF)) << 16)) & _M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """A 32-bit integer bijection (xorshift-multiply finaliser)."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


def _mix32_int(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    return x ^ (x >> 16)


def _key(seed: int, stream: int) -> int:
    return _mix32_int(_mix32_int(seed) ^ ((stream * 0x9E3779B9) & _M32))


_ROUND_KEYS = [_mix32_int(0xA5A5A5A5 + 0x61C88647 * r) for r in range(7)]
_CHUNK = 1 << 23


def _state(idx: torch.Tensor, key: int) -> torch.Tensor:
    lo = idx & _M32
    hi = idx >> 32
    return _mix32(lo ^ _mix32((hi + key) & _M32))


def counter_uniform(numel: int, seed: int, stream: int, offset: int = 0,
                    device="cpu") -> torch.Tensor:
    """int64 tensor of 32-bit uniform integers, element i = f(seed, stream, offset+i)."""
    out = torch.empty(numel, dtype=torch.int64, device=device)
    key = _key(seed, stream)
    for start in range(0, numel, _CHUNK):
        n = min(_CHUNK, numel - start)
        idx = torch.arange(offset + start, offset + start + n, dtype=torch.int64, device=device)
        out[start:start + n] = _mix32(_state(idx, key) ^ _ROUND_KEYS[6])
    return out


def counter_normal(numel: int, seed: int, stream: int, offset: int = 0,
                   device="cpu") -> torch.Tensor:
    """float32 tensor of approximately N(0,1) values (Irwin-Hall of 12 uniforms)."""
    out = torch.empty(numel, dtype=torch.float32, device=device)
    key = _key(seed, stream)
    for start in range(0, numel, _CHUNK):
        n = min(_CHUNK, numel - start)
        idx = torch.arange(offset + start, offset + start + n, dtype=torch.int64, device=device)
        st = _state(idx, key)
        acc = torch.zeros(n, dtype=torch.int64, device=device)
        for r in range(6):
            h = _mix32(st ^ _ROUND_KEYS[r])
            acc += (h & 0xFFFF) + (h >> 16)
        # 12 * 32767.5 = 393210; the difference is an integer below 2^24, so
        # the conversion and the division by 2^16 are exact in float32.
        out[start:start + n] = (acc - 393210).to(torch.float32) / 65536.0
    return out


def bf16_normal(shape, std: float, seed: int, stream: int, offset: int = 0,
                device="cpu", outlier_frac: float = 0.0, outlier_scale: float = 1.0,
                outlier_stream: int | None = None) -> torch.Tensor:
    """bfloat16 tensor ~ N(0, std^2), optionally with a seeded Bernoulli fraction of
    elements multiplied by ``outlier_scale``.  Identical on every device: the
    float32 multiplies are single IEEE roundings and the bf16 cast is RNE."""
    numel = int(np.prod(shape))
    z = counter_normal(numel, seed, stream, offset, device)
    z.mul_(torch.tensor(std, dtype=torch.float32, device=device))
    if outlier_frac > 0.0:
        u = counter_uniform(numel, seed, outlier_stream if outlier_stream is not None else stream + 1000,
                            offset, device)
        thresh = int(outlier_frac * 2.0 ** 32)
        sel = u < thresh
        z = torch.where(sel, z * torch.tensor(outlier_scale, dtype=torch.float32, device=device), z)
    return z.to(torch.bfloat16).reshape(shape)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
STREAM_X, STREAM_W13, STREAM_W2, STREAM_OUTLIER = 1, 2, 3, 4


@dataclass
class MoEConfig:
    name: str
    index: int
    E: int                 # local experts (c5: 256 routed + 1 shared)
    H: int                 # hidden
    I: int                 # expert intermediate
    layout: str            # "masked" | "contig"
    max_m: int = 0         # masked layout: rows per expert
    T: int = 0             # tokens (router configs)
    topk: int = 0
    n_global_experts: int = 0
    ep: int = 0            # expert-parallel group size the routing simulates
    tokens_per_rank: int = 0
    zipf_a: float = 1.1
    rows: int = 0          # contig: total token-rows
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    shared_expert: bool = False
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return 1000 + self.index


CONFIGS = {
    "c1": MoEConfig(
        "c1_tiny_masked", 0, E=4, H=256, I=128, layout="masked", max_m=128, T=64, topk=2,
        description="tiny MoE FFN, masked layout: E=4, hidden 256, intermediate 128, T=64, "
                    "top-2 from softmax of N(0,1) router logits"),
    "c2": MoEConfig(
        "c2_decode_ep72", 1, E=4, H=7168, I=2048, layout="masked", max_m=1024, topk=8,
        n_global_experts=288, ep=72, tokens_per_rank=256,
        description="DeepSeek-V3-shaped decode, EP72-like: 4 local experts, masked max_m=1024, "
                    "counts from 72x256 tokens, top-8 over 288 experts at Zipf(1.1)"),
    "c3": MoEConfig(
        "c3_prefill_ep32", 2, E=9, H=7168, I=2048, layout="contig", rows=32768, topk=1,
        outlier_frac=0.01, outlier_scale=20.0,
        description="DeepSeek-V3-shaped prefill, EP32-like: 9 local experts, contiguous layout, "
                    "32768 token-rows split Zipf(1.1), segments padded to 128, 1% outliers x20"),
    "c4": MoEConfig(
        "c4_decode_ep48", 3, E=6, H=7168, I=2048, layout="masked", max_m=2048, topk=8,
        n_global_experts=288, ep=48, tokens_per_rank=768,
        description="large-batch decode, 48-GPU domain: 6 local experts, masked max_m=2048, "
                    "counts from 48x768 tokens, top-8 over 288 experts at Zipf(1.1)"),
    "c5": MoEConfig(
        "c5_all_experts_decode", 4, E=257, H=7168, I=2048, layout="masked", max_m=128, T=64, topk=8,
        shared_expert=True,
        description="single-GPU decode layer: 256 routed experts + 1 shared, T=64, top-8 "
                    "from softmax of N(0,1) logits, masked layout"),
    # small-batch / latency regime of the same layer: 1, 4 or 16 tokens per
    # step (one decode token, multi-token-prediction-like drafts)
    "c5t1": MoEConfig(
        "c5t1_all_experts_decode_T1", 5, E=257, H=7168, I=2048, layout="masked", max_m=16, T=1, topk=8,
        shared_expert=True,
        description="single-GPU decode layer, latency regime: 256 routed experts + 1 shared, "
                    "T=1, top-8 from softmax of N(0,1) logits, masked max_m=16"),
    "c5t4": MoEConfig(
        "c5t4_all_experts_decode_T4", 6, E=257, H=7168, I=2048, layout="masked", max_m=16, T=4, topk=8,
        shared_expert=True,
        description="single-GPU decode layer, latency regime: 256 routed experts + 1 shared, "
                    "T=4, top-8 from softmax of N(0,1) logits, masked max_m=16"),
    "c5t16": MoEConfig(
        "c5t16_all_experts_decode_T16", 7, E=257, H=7168, I=2048, layout="masked", max_m=16, T=16, topk=8,
        shared_expert=True,
        description="single-GPU decode layer, latency regime: 256 routed experts + 1 shared, "
                    "T=16, top-8 from softmax of N(0,1) logits, masked max_m=16"),
}


def get_config(name: str) -> MoEConfig:
    return CONFIGS[name]


def zipf_split(total: int, parts: int, a: float) -> np.ndarray:
    """Split ``total`` rows over ``parts`` experts with p_r proportional to r^-a,
    rounded by the largest-remainder method (ties to the lower rank)."""
    p = np.arange(1, parts + 1, dtype=np.float64) ** (-a)
    p /= p.sum()
    raw = p * total
    base = np.floor(raw).astype(np.int64)
    rem = total - int(base.sum())
    order = np.argsort(-(raw - base), kind="stable")
    base[order[:rem]] += 1
    return base


def _softmax_topk(logits: np.ndarray, k: int):
    """Router stand-in: softmax over all experts (fp64), top-k by probability with
    ties to the lower id, weights renormalised to sum to one."""
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    pk = np.take_along_axis(p, order, axis=1)
    w = pk / pk.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def _zipf_routing(cfg: MoEConfig, rng: np.random.Generator):
    """Global routing of ep*tokens_per_rank tokens, each picking top-k distinct
    experts out of n_global_experts by Gumbel-top-k on Zipf(a) log-popularity.
    Expert ranks are mapped to ids by a seeded permutation.  The per-token
    weights are the softmax of the perturbed scores of the chosen experts."""
    n_tok = cfg.ep * cfg.tokens_per_rank
    n_exp = cfg.n_global_experts
    pop = np.arange(1, n_exp + 1, dtype=np.float64) ** (-cfg.zipf_a)
    pop /= pop.sum()
    rank_to_id = rng.permutation(n_exp)
    logp = np.empty(n_exp)
    logp[rank_to_id] = np.log(pop)
    gumbel = rng.gumbel(size=(n_tok, n_exp))
    score = logp[None, :] + gumbel
    ids = np.argsort(-score, axis=1, kind="stable")[:, :cfg.topk]
    sc = np.take_along_axis(score, ids, axis=1)
    sc = sc - sc.max(axis=1, keepdims=True)
    w = np.exp(sc)
    w /= w.sum(axis=1, keepdims=True)
    group = int(rng.integers(0, cfg.ep))
    return ids.astype(np.int32), w.astype(np.float32), group


def make_routing(cfg: MoEConfig) -> dict:
    """Routing for one config: token-order ``topk_ids`` (global expert ids),
    ``topk_w``, the local expert range, and bookkeeping for the report."""
    rng = np.random.default_rng(cfg.seed)
    if cfg.name.startswith("c1") or cfg.name.startswith("c5"):
        n_routed = cfg.E - (1 if cfg.shared_expert else 0)
        logits = rng.standard_normal((cfg.T, n_routed))
        ids, w = _softmax_topk(logits, cfg.topk)
        if cfg.shared_expert:
            # the shared expert is local expert n_routed; every token uses it at weight 1
            ids = np.concatenate([ids, np.full((cfg.T, 1), n_routed, np.int32)], axis=1)
            w = np.concatenate([w, np.ones((cfg.T, 1), np.float32)], axis=1)
        return dict(topk_ids=ids, topk_w=w, T=cfg.T, k=ids.shape[1], expert_begin=0,
                    E=cfg.E, global_tokens=cfg.T)
    if cfg.layout == "contig":
        counts = zipf_split(cfg.rows, cfg.E, cfg.zipf_a)
        assign = np.repeat(np.arange(cfg.E, dtype=np.int32), counts)
        assign = assign[rng.permutation(cfg.rows)]
        return dict(topk_ids=assign[:, None].copy(), topk_w=np.ones((cfg.rows, 1), np.float32),
                    T=cfg.rows, k=1, expert_begin=0, E=cfg.E, global_tokens=cfg.rows,
                    split=counts)
    ids, w, group = _zipf_routing(cfg, rng)
    eb = group * cfg.E
    local = ((ids >= eb) & (ids < eb + cfg.E)).any(axis=1)
    ids_l = ids[local]
    w_l = w[local]
    raw_counts = np.array([(ids_l == eb + e).sum() for e in range(cfg.E)], np.int64)
    return dict(topk_ids=np.ascontiguousarray(ids_l), topk_w=np.ascontiguousarray(w_l),
                T=int(local.sum()), k=cfg.topk, expert_begin=eb, E=cfg.E,
                global_tokens=ids.shape[0], raw_counts=raw_counts)


def make_activations(cfg: MoEConfig, T: int, device="cpu", row0: int = 0,
                     rows: int | None = None) -> torch.Tensor:
    """Token activations x [T, H] bf16 ~ N(0,1) (c3: 1% of elements x20).
    ``row0``/``rows`` regenerate a slice of rows alone."""
    rows = T - row0 if rows is None else rows
    return bf16_normal((rows, cfg.H), 1.0, cfg.seed, STREAM_X, offset=row0 * cfg.H,
                       device=device, outlier_frac=cfg.outlier_frac,
                       outlier_scale=cfg.outlier_scale, outlier_stream=STREAM_OUTLIER)


def make_expert_weights(cfg: MoEConfig, which: str, expert: int, device="cpu",
                        row0: int = 0, rows: int | None = None) -> torch.Tensor:
    """bf16 weights of one expert in K-major storage, std 1/sqrt(K):
    ``which='w13'`` -> [2I, H] (gate rows [0, I), then up rows [I, 2I));
    ``which='w2'``  -> [H, I].  ``row0``/``rows`` select a row slice."""
    if which == "w13":
        N, K, stream = 2 * cfg.I, cfg.H, STREAM_W13
    elif which == "w2":
        N, K, stream = cfg.H, cfg.I, STREAM_W2
    else:
        raise ValueError(which)
    rows = N - row0 if rows is None else rows
    off = expert * N * K + row0 * K
    return bf16_normal((rows, K), 1.0 / math.sqrt(K), cfg.seed, stream, offset=off, device=device)
