"""Seeded synthetic inputs for MoE FusedDispatch / FusedCombine.

This module only draws inputs: router logits, token activations, a
redundant-expert replica map and synthetic expert outputs.  It holds none of
the routing, quantization or combine arithmetic, so both the CUDA path and the
CPU oracle can be fed from it without sharing any of the method's code.

Workloads (CloudMatrix384 write-up, "Decode Phase" and "FusedDispatch and
FusedCombine"; StrataCL analysis, section 4.1 MoE dispatch/combine table):

* ``t64_h256_e8_k2``        64 tokens, hidden 256, 8 experts, top-2; identity experts.
* ``t96_h7168_e256_k8``     one decode local batch (96 tokens); 0.1 % of the
                            activations scaled x50 as outliers.
* ``t4096_h7168_e256p288_k8`` 4096 tokens, 256 logical experts plus 32 redundant
                            replicas (288 physical), Zipf(1.2) expert popularity.
* ``t16384_h2048_e64_k6``   16384 tokens, hidden 2048, 64 experts, top-6; expert
                            outputs N(0, 0.5); 10 back-to-back iterations.
* ``t30720_h7168_e256_k8``  global decode batch 96 x 320; Zipf(1.2) popularity;
                            buffers sized for worst-case per-expert capacity.

Every tensor comes from its own numpy PCG64 stream, derived from
``SeedSequence(seed, spawn_key=(stream_id,))``, so any one tensor can be redrawn
without drawing the others.  bf16 values are carried as ``uint16`` bit patterns
produced by round-to-nearest-even from the float32 draw.
"""
from __future__ import annotations

import dataclasses

import numpy as np

# Sub-stream ids: one per drawn tensor.
_S_X, _S_LOGITS, _S_EXOUT, _S_OUTLIER, _S_PERM = 1, 2, 3, 4, 5

_CHUNK = 1 << 24  # elements drawn per numpy call for large tensors


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens in the batch
    H: int            # hidden size
    E: int            # logical experts
    P: int            # physical expert slots (E plus redundant replicas)
    k: int            # experts per token
    x_sigma: float = 1.0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    zipf_s: float | None = None
    replicas: int = 0          # hot experts that get one extra replica
    ex_sigma: float = 1.0
    identity_experts: bool = False
    iterations: int = 1
    group: int = 128

    @property
    def G(self) -> int:
        return self.H // self.group

    @property
    def rows(self) -> int:
        return self.T * self.k

    def describe(self) -> str:
        """The synthetic inputs of a timed run, in words: the logits, the
        activations, the replica map and the expert rows combine reads."""
        logits = "N(0,1) logits" + (f" + Zipf({self.zipf_s:g}) expert bias" if self.zipf_s else "")
        x = f"N(0,{self.x_sigma:g}) bf16 x"
        if self.outlier_frac:
            x += f" with {100 * self.outlier_frac:g} % of elements x{self.outlier_scale:g}"
        parts = [logits, x]
        if self.replicas:
            parts.append(f"{self.replicas} hot experts with one extra replica")
        ex = f"N(0,{self.ex_sigma:g}) bf16 expert rows"
        if self.identity_experts:
            ex += " (identity experts in the parity runs)"
        parts.append(ex)
        return "synthetic (seeded; " + "; ".join(parts) + ")"

    def algorithmic_bytes(self) -> dict:
        """Bytes each call must move at least once (no re-reads, no padding).

        plan:     logits read, gates/slot/src_token written, counts/offsets.
        dispatch: x read once; each token's INT8 row and fp32 group scales
                  written k times; slot read.
        combine:  k bf16 expert rows read per token, gates and slot read,
                  y written once.
        """
        T, H, E, P, k, G = self.T, self.H, self.E, self.P, self.k, self.G
        plan = T * E * 4 + 3 * T * k * 4 + 2 * (P + 1) * 4
        dispatch = T * H * 2 + T * k * H + T * k * G * 4 + T * k * 4
        combine = T * k * H * 2 + T * k * 8 + T * H * 2
        return {"plan": plan, "dispatch": dispatch, "combine": combine,
                "total": plan + dispatch + combine}


WORKLOADS = {
    w.name: w
    for w in [
        Workload("t64_h256_e8_k2", T=64, H=256, E=8, P=8, k=2, identity_experts=True),
        Workload("t96_h7168_e256_k8", T=96, H=7168, E=256, P=256, k=8,
                 outlier_frac=0.001, outlier_scale=50.0),
        Workload("t4096_h7168_e256p288_k8", T=4096, H=7168, E=256, P=288, k=8,
                 zipf_s=1.2, replicas=32),
        Workload("t16384_h2048_e64_k6", T=16384, H=2048, E=64, P=64, k=6,
                 ex_sigma=0.5, iterations=10),
        Workload("t30720_h7168_e256_k8", T=30720, H=7168, E=256, P=256, k=8,
                 zipf_s=1.2),
    ]
}

BENCH_WORKLOAD = "t4096_h7168_e256p288_k8"


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(stream,))))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, n: int, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        z = rng.standard_normal(hi - lo, dtype=np.float32)
        if sigma != 1.0:
            z *= np.float32(sigma)
        out[lo:hi] = f32_to_bf16_bits(z)
    return out


def expert_popularity_rank(w: Workload, seed: int = 0) -> np.ndarray:
    """1-based popularity rank of each logical expert (1 = most popular)."""
    return _rng(seed, _S_PERM).permutation(w.E).astype(np.int64) + 1


def zipf_bias(w: Workload, seed: int = 0) -> np.ndarray:
    """Per-expert logit bias -s*ln(rank): the router then favours experts with
    a Zipf(s)-shaped popularity.  Zero when the workload has no skew."""
    if w.zipf_s is None:
        return np.zeros(w.E, dtype=np.float32)
    r = expert_popularity_rank(w, seed).astype(np.float64)
    return (-w.zipf_s * np.log(r)).astype(np.float32)


def make_logits(w: Workload, seed: int = 0, T: int | None = None) -> np.ndarray:
    """Router logits, float32 [T, E]: N(0,1) plus the Zipf bias if any."""
    T = w.T if T is None else T
    z = _rng(seed, _S_LOGITS).standard_normal((T, w.E), dtype=np.float32)
    return (z + zipf_bias(w, seed)[None, :]).astype(np.float32)


def make_x(w: Workload, seed: int = 0, T: int | None = None) -> np.ndarray:
    """Token activations, bf16 bits uint16 [T, H].

    With ``outlier_frac`` > 0, exactly round(frac*T*H) distinct element
    positions (a seeded draw without replacement) hold bf16(scale * z) instead
    of bf16(z)."""
    T = w.T if T is None else T
    n = T * w.H
    rng = _rng(seed, _S_X)
    if w.outlier_frac <= 0.0:
        return _normal_bf16(rng, n, w.x_sigma).reshape(T, w.H)
    z = rng.standard_normal(n, dtype=np.float32) * np.float32(w.x_sigma)
    n_out = int(round(w.outlier_frac * n))
    pos = _rng(seed, _S_OUTLIER).choice(n, size=n_out, replace=False)
    z[pos] *= np.float32(w.outlier_scale)
    return f32_to_bf16_bits(z).reshape(T, w.H)


def make_expert_out(w: Workload, seed: int = 0, rows: int | None = None) -> np.ndarray:
    """Synthetic expert outputs, bf16 bits uint16 [rows, H], N(0, ex_sigma) per
    slot row (rows defaults to T*k, one per dispatched copy)."""
    rows = w.rows if rows is None else rows
    return _normal_bf16(_rng(seed, _S_EXOUT), rows * w.H, w.ex_sigma).reshape(rows, w.H)


def make_replica_map(w: Workload, seed: int = 0):
    """Logical -> physical expert map as CSR (rep_off int32 [E+1], rep_ids int32 [P]).

    The ``replicas`` most popular experts each get one extra physical slot,
    numbered E + (rank - 1); every other expert keeps its own id.  Returns
    (None, None) when P == E (identity map)."""
    if w.P == w.E:
        return None, None
    assert w.P == w.E + w.replicas, "P must equal E + replicas"
    rank = expert_popularity_rank(w, seed)
    off = np.zeros(w.E + 1, dtype=np.int32)
    ids = []
    for e in range(w.E):
        mine = [e]
        if rank[e] <= w.replicas:
            mine.append(w.E + int(rank[e]) - 1)
        ids.extend(mine)
        off[e + 1] = off[e] + len(mine)
    return off, np.asarray(ids, dtype=np.int32)


def make_inputs(w: Workload, seed: int = 0, with_expert_out: bool = True) -> dict:
    rep_off, rep_ids = make_replica_map(w, seed)
    d = {"logits": make_logits(w, seed), "x": make_x(w, seed),
         "rep_off": rep_off, "rep_ids": rep_ids}
    if with_expert_out and not w.identity_experts:
        d["ex_out"] = make_expert_out(w, seed)
    return d


def small_variant(w: Workload, T: int, name_suffix: str = "_small") -> Workload:
    """Same H/E/P/k/distributions with fewer tokens (for oracle-sized parity)."""
    return dataclasses.replace(w, name=w.name + name_suffix, T=T)
