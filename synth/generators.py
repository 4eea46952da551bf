"""Seeded synthetic inputs for filtering-first constrained SID beam decoding.

This module only draws random data: catalogues of semantic IDs (SIDs), the
synthetic model tensors (per-step token tables C_s and output heads W_s) and
request vectors u.  It holds none of the decoding arithmetic, so both the CUDA
path and the CPU oracle can read the same arrays without sharing method code.

Every draw comes from a PCG64 stream keyed by (seed, purpose, step), so each
array is reproducible on its own and independent of the others.

Distribution readings (the configuration text writes "N(0, x)"): x is the
variance, as in the usual N(mu, sigma^2) notation.  Hence u, C_s ~ N(0, 1/d)
have std d^-1/2 and W_s ~ N(0, 1/sqrt(d)) has std d^-1/4.  The alternative
reading (std 1/sqrt(d) for W_s) is available through ``w_std="literal"``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_PURPOSE = {
    "catalogue": 1,
    "permute": 2,
    "u": 3,
    "C": 4,
    "W": 5,
    "zipf": 6,
    "level": 7,
    "deco": 8,
    "concept": 9,
}


def rng_for(seed: int, purpose: str, step: int = 0) -> np.random.Generator:
    """Independent PCG64 stream for (seed, purpose, step)."""
    return np.random.Generator(
        np.random.PCG64(np.random.SeedSequence([int(seed), _PURPOSE[purpose], int(step)])))


# ---------------------------------------------------------------------------
# storage conversions (bit-level, no method arithmetic)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round-to-nearest-even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# configurations
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Config:
    name: str
    L: int
    V: int
    d: int
    w_dtype: str          # "f32" | "bf16" | "f16"
    batch: int
    beam: int
    topk: int
    catalogue: str        # generator name
    n_items: int
    params: dict = field(default_factory=dict)


CONFIGS = {
    "tiny": Config("tiny", L=3, V=256, d=64, w_dtype="f32", batch=1, beam=8, topk=8,
                   catalogue="uniform", n_items=20_000),
    "mid_sparse": Config("mid_sparse", L=3, V=2048, d=256, w_dtype="f32", batch=32, beam=32,
                         topk=32, catalogue="zipf_hier", n_items=1_000_000,
                         params={"zipf_a": 1.1, "items_per_child": 8}),
    "sweep_v2048": Config("sweep_v2048", L=3, V=2048, d=256, w_dtype="bf16", batch=32, beam=64,
                          topk=64, catalogue="fixed_fanout", n_items=10_000_000),
    "sweep_v4096": Config("sweep_v4096", L=3, V=4096, d=256, w_dtype="bf16", batch=32, beam=64,
                          topk=64, catalogue="fixed_fanout", n_items=10_000_000),
    "sweep_v8192": Config("sweep_v8192", L=3, V=8192, d=256, w_dtype="bf16", batch=32, beam=64,
                          topk=64, catalogue="fixed_fanout", n_items=10_000_000),
    "sweep_v16384": Config("sweep_v16384", L=3, V=16384, d=256, w_dtype="bf16", batch=32, beam=64,
                           topk=64, catalogue="fixed_fanout", n_items=10_000_000),
    "dense_early": Config("dense_early", L=4, V=4096, d=384, w_dtype="f16", batch=128, beam=64,
                          topk=64, catalogue="dense_early", n_items=50_000_000,
                          params={"p_step2": 0.9}),
    "large": Config("large", L=4, V=8192, d=512, w_dtype="bf16", batch=64, beam=256, topk=256,
                    catalogue="zipf_geometric", n_items=100_000_000,
                    params={"zipf_a": 1.05, "decay": 0.25}),
}


# ---------------------------------------------------------------------------
# catalogue helpers
# ---------------------------------------------------------------------------

def _even_split(total: np.ndarray, parts: np.ndarray) -> np.ndarray:
    """Split total[g] items over parts[g] children as evenly as possible.

    Returns the per-child counts, group-major; the first (total % parts)
    children of a group get one extra item."""
    total = np.asarray(total, np.int64)
    parts = np.asarray(parts, np.int64)
    base = np.repeat(total // parts, parts)
    rem = np.repeat(total % parts, parts)
    starts = np.cumsum(parts) - parts
    pos = np.arange(parts.sum(), dtype=np.int64) - np.repeat(starts, parts)
    return base + (pos < rem)


def distinct_per_group(rng: np.random.Generator, counts: np.ndarray, V: int) -> np.ndarray:
    """For each group g draw counts[g] distinct values uniformly from [0, V).

    Returns a flat int64 array, group-major, ascending within each group.
    Small groups use rejection of repeated values (the procedure treats all
    values alike, so the resulting subset is uniform); groups larger than V/8
    take a prefix of a random permutation."""
    counts = np.asarray(counts, np.int64)
    if counts.size == 0:
        return np.zeros(0, np.int64)
    if (counts > V).any() or (counts < 0).any():
        raise ValueError("group asks for more distinct values than V")
    out = np.empty(int(counts.sum()), np.int64)
    starts = np.cumsum(counts) - counts
    big = counts > max(V // 8, 1)
    for g in np.nonzero(big)[0]:
        k = int(counts[g])
        out[starts[g]:starts[g] + k] = np.sort(rng.permutation(V)[:k])
    small = np.nonzero(~big & (counts > 0))[0]
    if small.size:
        sc = counts[small]
        gid = np.repeat(np.arange(small.size, dtype=np.int64), sc)
        vals = rng.integers(0, V, size=gid.size, dtype=np.int64)
        active = np.arange(gid.size, dtype=np.int64)      # positions still checked
        while True:
            key = gid[active] * V + vals[active]
            order = np.argsort(key, kind="stable")
            ks = key[order]
            dup = np.zeros(ks.size, bool)
            dup[1:] = ks[1:] == ks[:-1]
            if not dup.any():
                break
            redo = active[order[dup]]
            vals[redo] = rng.integers(0, V, size=redo.size, dtype=np.int64)
            # only groups that saw a repeat need checking again
            bad = np.zeros(small.size, bool)
            bad[gid[redo]] = True
            active = np.nonzero(bad[gid])[0]
        key = gid * V + vals
        key.sort()
        sv = key - gid * V
        sstarts = starts[small]
        dst = np.repeat(sstarts, sc) + (np.arange(gid.size) - np.repeat(np.cumsum(sc) - sc, sc))
        out[dst] = sv
    return out


def _zipf_probs(V: int, a: float) -> np.ndarray:
    r = np.arange(1, V + 1, dtype=np.float64)
    p = r ** (-a)
    return p / p.sum()


def _shuffle_rows(sids: np.ndarray, seed: int) -> np.ndarray:
    perm = rng_for(seed, "permute").permutation(sids.shape[0])
    return np.ascontiguousarray(sids[perm])


def _hier(seed: int, V: int, top_tokens: np.ndarray, top_items: np.ndarray, child_counts):
    """Top-down budget generator.

    top_tokens/top_items: step-1 tokens and their item budgets.
    child_counts: list, one per lower level except the leaf level, of
    functions items -> number of distinct children.  Each prefix splits its
    items evenly over its children; at the leaf level each prefix gets as
    many distinct leaves as it has items."""
    levels_tok = [top_tokens.astype(np.int64)]
    items = top_items.astype(np.int64)
    per_level_items = [items]
    for lvl, fn in enumerate(child_counts):
        k = fn(items)
        k = np.minimum(np.maximum(k, 1), V)
        k = np.minimum(k, items)
        child = distinct_per_group(rng_for(seed, "level", 2 + lvl), k, V)
        items = _even_split(items, k)
        levels_tok.append(child)
        per_level_items.append(items)
    # leaf level: one distinct token per item
    if (items > V).any():
        raise ValueError("a prefix holds more items than the codebook allows")
    leaf = distinct_per_group(rng_for(seed, "level", 9), items, V)
    levels_tok.append(leaf)
    # counts of items under each token of each level
    cols = []
    for li, tok in enumerate(levels_tok[:-1]):
        cols.append(np.repeat(tok, per_level_items[li]))
    cols.append(leaf)
    return np.stack(cols, axis=1).astype(np.int32)


# ---------------------------------------------------------------------------
# catalogue generators
# ---------------------------------------------------------------------------

def catalogue_uniform(L: int, V: int, n: int, seed: int) -> np.ndarray:
    """n distinct SIDs drawn uniformly without replacement from [0, V)^L."""
    space = V ** L
    if n > space:
        raise ValueError("more items than SIDs")
    rng = rng_for(seed, "catalogue")
    flat = rng.choice(space, size=n, replace=False)
    out = np.empty((n, L), np.int32)
    for s in range(L - 1, -1, -1):
        out[:, s] = flat % V
        flat = flat // V
    return out


def catalogue_zipf_hier(V: int, n: int, seed: int, zipf_a: float = 1.1,
                        items_per_child: int = 8) -> np.ndarray:
    """L=3 hierarchical catalogue: step-1 token budgets ~ Multinomial(n, Zipf(a)),
    each step-1 token has clamp(round(n_t/items_per_child), 1, V) distinct
    children, each 2-prefix has as many distinct leaves as items."""
    p = _zipf_probs(V, zipf_a)
    n_rank = rng_for(seed, "zipf").multinomial(n, p)
    perm = rng_for(seed, "zipf", 1).permutation(V)          # rank -> token
    n_tok = np.zeros(V, np.int64)
    n_tok[perm] = n_rank
    toks = np.nonzero(n_tok)[0]
    sids = _hier(seed, V, toks, n_tok[toks],
                 [lambda it: np.rint(it / items_per_child).astype(np.int64)])
    return _shuffle_rows(sids, seed)


def catalogue_fixed_fanout(V: int, n: int, seed: int, f1: int = 2048, f2: int = 64) -> np.ndarray:
    """L=3 catalogue with constant fan-out across V: f1 distinct step-1 tokens,
    f2 children each, and the remaining budget spread as evenly as possible
    over the 2-prefixes (the first ones get one extra leaf)."""
    f1 = min(f1, V)
    t1 = np.sort(rng_for(seed, "catalogue").permutation(V)[:f1])
    k2 = np.full(f1, f2, np.int64)
    t2 = distinct_per_group(rng_for(seed, "level", 2), k2, V)
    n2 = f1 * f2
    leaves_per = np.full(n2, n // n2, np.int64)
    leaves_per[: n % n2] += 1
    t3 = distinct_per_group(rng_for(seed, "level", 9), leaves_per, V)
    items_per_t1 = np.add.reduceat(leaves_per, np.arange(0, n2, f2))
    col1 = np.repeat(t1, items_per_t1)
    col2 = np.repeat(t2, leaves_per)
    sids = np.stack([col1, col2, t3], axis=1).astype(np.int32)
    return _shuffle_rows(sids, seed)


def catalogue_dense_early(V: int, n: int, seed: int, p_step2: float = 0.9) -> np.ndarray:
    """L=4 catalogue whose first two steps are nearly dense.

    Step 1: every token is legal.  Step 2: every token is legal under each
    step-1 token independently with probability p_step2 (so the fan-out is
    Binomial(V, p_step2)).  Steps 3 and 4: fan-outs 1+Poisson(l3) and
    1+Poisson(l4) with l3 = 3*l4, l4 chosen so the expected item count is n."""
    rng = rng_for(seed, "catalogue")
    mask = rng.random((V, V)) < p_step2
    t1_idx, t2 = np.nonzero(mask)                 # row-major: sorted by (t1, t2)
    n2 = t1_idx.size
    per2 = n / n2                                  # items per 2-prefix
    # (1 + 3x)(1 + x) = per2  ->  3x^2 + 4x + (1 - per2) = 0
    x = (-4.0 + math.sqrt(16.0 - 12.0 * (1.0 - per2))) / 6.0
    l3, l4 = 3.0 * x, x
    k3 = np.minimum(1 + rng_for(seed, "level", 3).poisson(l3, size=n2), V)
    t3 = distinct_per_group(rng_for(seed, "level", 4), k3, V)
    n3 = t3.size
    k4 = np.minimum(1 + rng_for(seed, "level", 5).poisson(l4, size=n3), V)
    t4 = distinct_per_group(rng_for(seed, "level", 6), k4, V)
    # assemble
    items3 = k4
    items2 = np.add.reduceat(items3, np.cumsum(k3) - k3)
    col1 = np.repeat(t1_idx, items2)
    col2 = np.repeat(t2, items2)
    col3 = np.repeat(t3, items3)
    sids = np.stack([col1, col2, col3, t4], axis=1).astype(np.int32)
    return _shuffle_rows(sids, seed)


def catalogue_zipf_geometric(V: int, n: int, seed: int, zipf_a: float = 1.05,
                             decay: float = 0.25) -> np.ndarray:
    """L=4 catalogue: Zipf(a) step-1 budgets and geometric fan-out decay.

    Mean fan-outs f2, f3 = decay*f2, f4 = decay*f3 with f2*f3*f4 = n/V.  Each
    prefix with m items takes clamp(round(m / (f3*f4)), 1, V) children at
    step 2 and clamp(round(m / f4), 1, V) at step 3; leaves are distinct."""
    per_t1 = n / V
    f2 = (per_t1 / decay ** 3) ** (1.0 / 3.0)
    f3 = decay * f2
    f4 = decay * f3
    p = _zipf_probs(V, zipf_a)
    n_rank = rng_for(seed, "zipf").multinomial(n, p)
    perm = rng_for(seed, "zipf", 1).permutation(V)
    n_tok = np.zeros(V, np.int64)
    n_tok[perm] = n_rank
    toks = np.nonzero(n_tok)[0]
    sids = _hier(seed, V, toks, n_tok[toks],
                 [lambda it: np.rint(it / (f3 * f4)).astype(np.int64),
                  lambda it: np.rint(it / f4).astype(np.int64)])
    return _shuffle_rows(sids, seed)


def product_catalogue(L: int, V: int) -> np.ndarray:
    """Every SID of [0, V)^L (the full product space), lexicographic order."""
    grids = np.meshgrid(*([np.arange(V)] * L), indexing="ij")
    return np.stack([g.reshape(-1) for g in grids], axis=1).astype(np.int32)


def make_catalogue(cfg: Config, seed: int = 0) -> np.ndarray:
    if cfg.catalogue == "uniform":
        return catalogue_uniform(cfg.L, cfg.V, cfg.n_items, seed)
    if cfg.catalogue == "zipf_hier":
        return catalogue_zipf_hier(cfg.V, cfg.n_items, seed, **cfg.params)
    if cfg.catalogue == "fixed_fanout":
        return catalogue_fixed_fanout(cfg.V, cfg.n_items, seed)
    if cfg.catalogue == "dense_early":
        return catalogue_dense_early(cfg.V, cfg.n_items, seed, **cfg.params)
    if cfg.catalogue == "zipf_geometric":
        return catalogue_zipf_geometric(cfg.V, cfg.n_items, seed, **cfg.params)
    raise KeyError(cfg.catalogue)


# ---------------------------------------------------------------------------
# model tensors and requests
# ---------------------------------------------------------------------------

@dataclass
class SynthModel:
    L: int
    V: int
    d: int
    w_dtype: str
    C: list            # L-1 float32 arrays [V, d]: C[s] is added after choosing a step-(s+1) token
    W: list            # L arrays [V, d]: float32, float16, or uint16 bfloat16 bit patterns

    def W_as_f64(self, s: int) -> np.ndarray:
        """Stored weights of step s (0-based) widened exactly to float64."""
        w = self.W[s]
        if self.w_dtype == "bf16":
            return bf16_bits_to_f32(w).astype(np.float64)
        return np.asarray(w).astype(np.float64)


def make_model(L: int, V: int, d: int, w_dtype: str = "f32", seed: int = 0,
               w_std: str = "variance") -> SynthModel:
    """C_s ~ N(0, 1/d) (variance) in float32; W_s ~ N(0, 1/sqrt(d)) (variance),
    rounded to w_dtype."""
    c_std = 1.0 / math.sqrt(d)
    w_sd = d ** -0.25 if w_std == "variance" else 1.0 / math.sqrt(d)
    C = [(rng_for(seed, "C", s).standard_normal((V, d)) * c_std).astype(np.float32)
         for s in range(L - 1)]
    W = []
    for s in range(L):
        w32 = (rng_for(seed, "W", s).standard_normal((V, d)) * w_sd).astype(np.float32)
        if w_dtype == "f32":
            W.append(w32)
        elif w_dtype == "bf16":
            W.append(f32_to_bf16_bits(w32))
        elif w_dtype == "f16":
            W.append(w32.astype(np.float16))
        else:
            raise ValueError(w_dtype)
    return SynthModel(L, V, d, w_dtype, C, W)


def make_requests(B: int, d: int, seed: int = 0) -> np.ndarray:
    """Request vectors u ~ N(0, 1/d) (variance), float32 [B, d]."""
    return (rng_for(seed, "u").standard_normal((B, d)) / math.sqrt(d)).astype(np.float32)


# ---------------------------------------------------------------------------
# light decoder (the model producing each step's hidden vector from a fixed
# set of concept vectors and the prefix of chosen tokens)
# ---------------------------------------------------------------------------

@dataclass
class DecoWeights:
    """Random weights of a causal decoder of `layers` layers, width d, `heads`
    attention heads and MLP width `ffn`, for an L-step SID decode with M
    concept vectors.  Every matrix is float32 [out][in] (row-major).
      E[s]: [V, d] embedding of the token chosen at step s+1 (s = 0..L-2)
      P:    [M + L - 1, d] position embeddings
      Wq, Wk, Wv, Wo: per layer [d, d];  W1: per layer [ffn, d];  W2: per layer [d, ffn]"""
    M: int
    d: int
    heads: int
    ffn: int
    layers: int
    E: list
    P: np.ndarray
    Wq: list
    Wk: list
    Wv: list
    Wo: list
    W1: list
    W2: list


def make_deco(L: int, V: int, d: int = 256, M: int = 2, heads: int = 4, ffn: int = 1024, layers: int = 2,
              seed: int = 0, zero_residual: bool = False) -> DecoWeights:
    """Embeddings ~ N(0, 1/d); projections ~ N(0, 1/fan_in) (variance), so
    activations stay of order one.  zero_residual: attention-output and
    MLP-output weights all zero (every layer leaves its input unchanged)."""
    def draw(i, shape, fan_in):
        return (rng_for(seed, "deco", i).standard_normal(shape) / math.sqrt(fan_in)).astype(np.float32)
    E = [draw(s, (V, d), d) for s in range(L - 1)]
    P = draw(10, (M + L - 1, d), d)
    Wq, Wk, Wv, Wo, W1, W2 = [], [], [], [], [], []
    for l in range(layers):
        b = 100 + 10 * l
        Wq.append(draw(b, (d, d), d))
        Wk.append(draw(b + 1, (d, d), d))
        Wv.append(draw(b + 2, (d, d), d))
        Wo.append(np.zeros((d, d), np.float32) if zero_residual else draw(b + 3, (d, d), d))
        W1.append(draw(b + 4, (ffn, d), d))
        W2.append(np.zeros((d, ffn), np.float32) if zero_residual else draw(b + 5, (d, ffn), ffn))
    return DecoWeights(M, d, heads, ffn, layers, E, P, Wq, Wk, Wv, Wo, W1, W2)


def make_concepts(B: int, M: int, d: int, seed: int = 0) -> np.ndarray:
    """Concept vectors of each request ~ N(0, 1/d) (variance), float32 [B, M, d]."""
    return (rng_for(seed, "concept").standard_normal((B, M, d)) / math.sqrt(d)).astype(np.float32)
