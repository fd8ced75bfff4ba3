"""Seeded synthetic workloads for block-sparse decode attention.

This module only makes inputs. It holds none of the arithmetic of the method
(no digests, scores, selection, attention or merge): the fp64 oracle and the
CUDA library both consume what it produces, and neither imports the other.

Random numbers come from one counter-based generator, defined here and, with
the same definition, in ``gen.cu`` for large device-side tensors:

* ``mix64`` is the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).
* element ``i`` of tensor stream ``s`` under seed ``seed`` takes three words
  ``mix64(key + 3 i + r)``, ``r = 0, 1, 2``, with ``key = mix64(mix64(seed) ^ s)``;
  the twelve 16-bit fields of those words, summed as integers, give an
  Irwin-Hall(12) variate ``z = sum / 65536 - 6``, which is exact in fp32,
  so the host and the device produce identical bits.
* a scaled value is ``fp32(z * sigma)`` (one IEEE multiply), optionally plus one
  IEEE add, then rounded to bf16 with round-to-nearest-even.

bf16 tensors are carried on the host as ``uint16`` bit patterns.

The workload shapes follow the decode workloads the paper evaluates
(ScoutAttention, arXiv HTML mirror, section 4 "Evaluation": Qwen3-8B and
Qwen3-14B, sparse budget 2048 tokens, block size 32, contexts up to 64K;
section 2.3: about 4 KB of KV per token per layer, i.e. 8 KV heads x 128 dims
x K and V x bf16).  They stand in for the LongBench prompts the paper uses,
which are not reproduced here.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# ---------------------------------------------------------------------------
# counter-based generator (bit-identical to gen.cu)
# ---------------------------------------------------------------------------
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor stream identifiers
STREAM_K = 1
STREAM_V = 2
STREAM_Q = 3
STREAM_X = 4
STREAM_W = 5
STREAM_QPRED = 6
STREAM_OCPU = 7
STREAM_LSECPU = 8
STREAM_WALK = 9


def mix64(x):
    """SplitMix64 output function on uint64 scalars or arrays (wrapping)."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    return mix64(mix64(np.uint64(seed)) ^ np.uint64(stream))


def irwin_hall(seed: int, stream: int, idx) -> np.ndarray:
    """Standard-ish normal variates (Irwin-Hall of 12 u16 fields), fp32, exact."""
    idx = np.asarray(idx, dtype=np.uint64)
    key = stream_key(seed, stream)
    total = np.zeros(idx.shape, dtype=np.int64)
    m16 = np.uint64(0xFFFF)
    with np.errstate(over="ignore"):
        base = key + np.uint64(3) * idx
        for r in range(3):
            h = mix64(base + np.uint64(r))
            for sh in (0, 16, 32, 48):
                total += ((h >> np.uint64(sh)) & m16).astype(np.int64)
    z = total.astype(np.float32) / np.float32(65536.0) - np.float32(6.0)
    return z.astype(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, stream: int, shape, sigma: float = 1.0, offset: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    z = irwin_hall(seed, stream, np.arange(offset, offset + n, dtype=np.uint64))
    return f32_to_bf16(z * np.float32(sigma)).reshape(shape)


def normal_f32(seed: int, stream: int, shape, sigma: float = 1.0, offset: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    z = irwin_hall(seed, stream, np.arange(offset, offset + n, dtype=np.uint64))
    return (z * np.float32(sigma)).reshape(shape)


# ---------------------------------------------------------------------------
# workload description
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Shape:
    """One decode-step workload for one layer.

    ``k`` is the budget in blocks per KV head (budget tokens / P).
    ``seq_lens`` (optional) gives ragged per-sequence lengths <= ``T``.
    """

    name: str
    B: int
    Hq: int
    Hkv: int
    T: int
    P: int
    k: int
    resident_frac: float
    kind: str = "minmax"  # or "mean"
    D: int = 128
    hidden: int = 0  # GEMM K (0: no GEMM in this workload)
    seed: int = 0
    heavy_frac: float = 0.05
    n_outliers: int = 4
    outlier_scale: float = 8.0
    heavy_gain: float = 3.0
    w_sigma: float = 0.02
    seq_lens: tuple | None = None

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def nblk(self) -> int:
        return -(-self.T // self.P)

    @property
    def units(self) -> int:
        return self.B * self.Hkv

    @property
    def words(self) -> int:
        return -(-self.nblk // 32)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def lens(self) -> np.ndarray:
        if self.seq_lens is None:
            return np.full(self.B, self.T, dtype=np.int32)
        s = np.asarray(self.seq_lens, dtype=np.int32)
        assert s.shape == (self.B,) and s.max() <= self.T and s.min() >= 0
        return s


def tiny() -> Shape:
    """Single-layer decode step: B=1, 8/2 heads, T=4096, P=32, top-16, 50% resident."""
    return Shape("tiny_b1_h8_t4k", B=1, Hq=8, Hkv=2, T=4096, P=32, k=16, resident_frac=0.5, hidden=1024)


def qwen3_8b() -> Shape:
    """Qwen3-8B-shaped layer: hidden 4096, 32/8 heads, B=8, T=16K, budget 2048, 25% resident."""
    return Shape("qwen3_8b_b8_t16k", B=8, Hq=32, Hkv=8, T=16384, P=32, k=64, resident_frac=0.25, hidden=4096)


def qwen3_14b() -> Shape:
    """Qwen3-14B-shaped layer: hidden 5120, 40/8 heads, B=40, T=32K, budget 2048, 25% resident."""
    return Shape("qwen3_14b_b40_t32k", B=40, Hq=40, Hkv=8, T=32768, P=32, k=64, resident_frac=0.25, hidden=5120)


def stress(P: int, budget: int, kind: str) -> Shape:
    """Stress point on the Qwen3-14B head shapes: B=4, T=128K."""
    return Shape(f"stress_p{P}_b{budget}_{kind}", B=4, Hq=40, Hkv=8, T=131072, P=P, k=budget // P,
                 resident_frac=0.25, kind=kind, hidden=0)


CONFIGS = {"tiny": tiny, "qwen3_8b": qwen3_8b, "qwen3_14b": qwen3_14b}


# ---------------------------------------------------------------------------
# structural metadata (small; computed once on the host, shared by both sides)
# ---------------------------------------------------------------------------
class Workload:
    """Seeded inputs of one :class:`Shape`.

    Logical tensors (host, bf16 bits as uint16):
      q        [B][Hq][D]         true query, N(0,1)
      K, V     [B][Hkv][T][D]     generated per unit on demand (``unit_kv``)
      X        [B][hidden]        layer input for the Q_pred GEMM, N(0,1)
      W        [Hq*D][hidden]     W_Q, N(0, w_sigma^2)
    Structure (shared by host and device):
      outliers         4 channel indices scaled by ``outlier_scale`` in K and V
      heavy[u][j]      5% of valid blocks per unit whose keys add heavy_gain * qhat_g
      hdir[u][D]       fp32(heavy_gain * qhat_g), qhat_g = normalize(sum_{h in g} q_h)
      resident[u][j]   seeded residency: round(frac * valid) blocks per unit
      page_table[u][j] slot of block j of unit u in the K/V pool (a seeded permutation)
    """

    def __init__(self, shape: Shape, pool_slots: int | None = None):
        """``pool_slots`` (profiling only) shrinks the K/V pool: blocks share slots, so
        the pool no longer holds each block's own keys and parity does not apply."""
        self.s = s = shape
        rng = np.random.Generator(np.random.PCG64(s.seed))
        self.seq_len = s.lens()
        self.outliers = np.sort(rng.choice(s.D, size=s.n_outliers, replace=False)).astype(np.int32)
        chan = np.ones(s.D, dtype=np.float32)
        chan[self.outliers] = np.float32(s.outlier_scale)
        self.chan_scale = chan
        self.q = normal_bf16(s.seed, STREAM_Q, (s.B, s.Hq, s.D))
        nvalid = -(-self.seq_len.astype(np.int64) // s.P)
        self.nvalid = nvalid.astype(np.int32)
        U, nb = s.units, s.nblk
        heavy = np.zeros((U, nb), dtype=np.uint8)
        resident = np.zeros((U, nb), dtype=np.uint8)
        for u in range(U):
            nv = int(nvalid[u // s.Hkv])
            if nv == 0:
                continue
            nh = int(round(s.heavy_frac * nv))
            if nh:
                heavy[u, rng.choice(nv, size=nh, replace=False)] = 1
            nr = int(round(s.resident_frac * nv))
            if nr:
                resident[u, rng.choice(nv, size=nr, replace=False)] = 1
        self.heavy = heavy
        self.resident = resident
        # heavy direction per unit: fp32(gain * normalize(sum of the group's query heads))
        qf = bf16_to_f32(self.q).astype(np.float64).reshape(s.B, s.Hkv, s.G, s.D)
        qs = qf.sum(axis=2)
        nrm = np.linalg.norm(qs, axis=-1, keepdims=True)
        nrm[nrm == 0] = 1.0
        self.hdir = (s.heavy_gain * qs / nrm).astype(np.float32).reshape(U, s.D)
        # pool slots: a seeded permutation so the page table is exercised
        nslots = U * nb
        perm = rng.permutation(nslots).astype(np.int32)
        if pool_slots is not None and pool_slots < nslots:
            perm = perm % np.int32(pool_slots)
            nslots = int(pool_slots)
        self.page_table = perm.reshape(U, nb)
        inv = np.empty(nslots, dtype=np.int32)
        inv[perm] = np.arange(U * nb, dtype=np.int32)
        self.slot_owner = inv  # slot -> u * nblk + j (one owner per slot)
        self.n_slots = nslots
        self.aliased = nslots < U * nb

    # -- bitmaps -----------------------------------------------------------
    def resident_bits(self, resident: np.ndarray | None = None) -> np.ndarray:
        """uint32 [B][Hkv][words], bit j%32 of word j//32 = block j resident."""
        s = self.s
        r = self.resident if resident is None else resident
        out = np.zeros((s.units, s.words), dtype=np.uint32)
        for j in range(s.nblk):
            out[:, j // 32] |= (r[:, j].astype(np.uint32) << np.uint32(j % 32))
        return out.reshape(s.B, s.Hkv, s.words)

    # -- logical K/V of one unit --------------------------------------------
    def unit_kv(self, u: int, which: str = "K") -> np.ndarray:
        """bf16 bits [nblk*P][D] of K or V of unit u = b * Hkv + kvh (logical token order).

        Element (t, d) of unit u is counter ``(u * nblk * P + t) * D + d`` of the
        K (or V) stream; tokens past ``seq_len`` exist but are never attended.
        """
        s = self.s
        Tp = s.nblk * s.P
        stream = STREAM_K if which == "K" else STREAM_V
        off = u * Tp * s.D
        z = irwin_hall(s.seed, stream, np.arange(off, off + Tp * s.D, dtype=np.uint64)).reshape(Tp, s.D)
        x = z * self.chan_scale[None, :]
        if which == "K":
            hv = np.repeat(self.heavy[u].astype(bool), s.P)
            x[hv] = x[hv] + self.hdir[u][None, :]
        return f32_to_bf16(x)

    # -- GEMM operands ------------------------------------------------------
    def gemm_x(self) -> np.ndarray:
        s = self.s
        return normal_bf16(s.seed, STREAM_X, (s.B, s.hidden))

    def gemm_w(self, rows: slice | None = None) -> np.ndarray:
        s = self.s
        N = s.Hq * s.D
        if rows is None:
            return normal_bf16(s.seed, STREAM_W, (N, s.hidden), sigma=s.w_sigma)
        r0, r1 = rows.start, rows.stop
        return normal_bf16(s.seed, STREAM_W, (r1 - r0, s.hidden), sigma=s.w_sigma, offset=r0 * s.hidden)

    # -- multi-step query walk ----------------------------------------------
    def walk(self, steps: int, cosine: float = 0.93, noise: float = 0.3):
        """True and predicted queries of decode steps 0 .. steps-1, bf16 bits [steps][B][Hq][D].

        q_0 is ``self.q``; q_t = sqrt(D) * normalize(q^_{t-1} + noise * n_t / sqrt(D)) with n_t
        ~ N(0, I) and q^ the unit vector (a step cosine near 0.96), rounded to bf16 each step.  Q_pred_t has the norm
        of q_t and cosine ``cosine`` to it: ||q_t|| (c q^_t + sqrt(1 - c^2) w_t) with w_t a
        seeded unit vector orthogonal to q_t.  (Table 1 of the pages gives cosines 0.93-0.97
        between predicted and true queries; the sweep uses the smallest.)
        """
        s = self.s
        n = s.B * s.Hq * s.D
        sqd = np.sqrt(np.float64(s.D))
        q = bf16_to_f32(self.q).astype(np.float64).reshape(s.B, s.Hq, s.D)
        qs, ps = [], []
        for t in range(steps):
            if t > 0:
                z = irwin_hall(s.seed, STREAM_WALK, np.arange(t * n, (t + 1) * n, dtype=np.uint64))
                q = q / np.linalg.norm(q, axis=-1, keepdims=True) + noise * z.astype(np.float64).reshape(q.shape) / sqd
                q = sqd * q / np.linalg.norm(q, axis=-1, keepdims=True)
                q = bf16_to_f32(f32_to_bf16(q.astype(np.float32))).astype(np.float64)
            qh = q / np.linalg.norm(q, axis=-1, keepdims=True)
            w = irwin_hall(s.seed, STREAM_QPRED, np.arange(t * n, (t + 1) * n, dtype=np.uint64))
            w = w.astype(np.float64).reshape(q.shape)
            w = w - (w * qh).sum(-1, keepdims=True) * qh
            w = w / np.linalg.norm(w, axis=-1, keepdims=True)
            pred = np.linalg.norm(q, axis=-1, keepdims=True) * (cosine * qh + np.sqrt(1.0 - cosine ** 2) * w)
            qs.append(f32_to_bf16(q.astype(np.float32)))
            ps.append(f32_to_bf16(pred.astype(np.float32)))
        return np.stack(qs), np.stack(ps)

    # -- CPU-side partial (stands in for the CPU worker's output) -----------
    def cpu_partial(self):
        """(O_cpu fp32 [B][Hq][D], LSE_cpu fp32 [B][Hq]) drawn from the generator."""
        s = self.s
        o = normal_f32(s.seed, STREAM_OCPU, (s.B, s.Hq, s.D), sigma=0.5)
        lse = normal_f32(s.seed, STREAM_LSECPU, (s.B, s.Hq), sigma=2.0) + np.float32(4.0)
        return o, lse
