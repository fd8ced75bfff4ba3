"""fp64 CPU oracle for GPU-CPU collaborative block-sparse decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The CUDA library never calls it, and it shares no code with the CUDA
library; inputs come from ``block_sparse_kv_pred_gb300.workload`` (bf16 bit
patterns as uint16), which holds none of the method's arithmetic.

Every quantity is computed in float64 from the exact bf16 input values, in the
order the paper states the method, with no blocking or fusion.  Sources (all
on the paper "ScoutAttention: Efficient KV Cache Offloading via Layer-Ahead
CPU Pre-computation for LLM Inference", arXiv 2603.27138):

* arXiv HTML, section 2.2 (block-wise sparse attention): the KV cache is cut
  into fixed-size blocks, each summarised by a digest; Quest's digest is the
  channel-wise min and max of K over the block, MoBA's the mean of K; the
  top-k blocks are chosen by the dot product of the query with the digests.
* arXiv HTML, section 3.2 (GPU-CPU collaborative block-wise sparse attention):
  the GPU scores every digest, takes the top-k blocks, attends the selected
  blocks that live in GPU memory, the CPU attends the selected blocks that do
  not, and the two partial results are combined with the FlashAttention /
  online-softmax rule.
* arXiv HTML, section 3.3 (layer-ahead CPU pre-computation) and Algorithm 1:
  Q_pred^{i+1} = W_Q^{i+1} X^i; B_pred = TopK(Q_pred K_digest^T);
  B_cpu = B_pred minus B_gpu; A = MERGE(A_gpu, A_cpu).
* arXiv HTML, section 3.4 (asynchronous periodic recall): important blocks are
  periodically copied back into GPU memory; each layer's recall interval is the
  largest number of decoding steps that keeps its CPU compute ratio (CPU tokens
  over the sparse budget) below a threshold beta, 12% by default, read from an
  offline profile.

Readings where the pages are silent (listed again in the design notes):
* GQA: query head h reads KV head h // G; one selection per (sequence, KV head),
  scored by the maximum over the G query heads of the group (the sum is a variant).
* Top-k order: score descending, ties to the lower block index; k_eff =
  min(k, number of valid blocks); lists are returned in ascending block order.
* The GPU partial attends S intersect R (the resident part of the top-k set); attending
  every resident block is a variant (parity unpinned: a reading).
* LSE is the natural log of sum exp(scale * q.k); partial outputs are normalised;
  an empty set gives O = 0, LSE = -inf.
* Tokens t >= seq_len are never attended and never enter a digest.
* Recall interval: every profiled step of the interval is strictly below beta;
  the interval is at least one step and at most the profiled length.
* Residency per page (one block of a sequence for all KV heads): a page is needed
  when any head selects it and ranked by the largest of its heads' scores (parity
  unpinned: the pages do not say how per-head selections map to shared pages).
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = -math.inf


# ---------------------------------------------------------------------------
# bf16 bit patterns
# ---------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even); returns uint16 bits."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1
    r = np.ldexp(np.rint(m * 256.0), e - 8)  # 8 significant bits, half-to-even
    f = r.astype(np.float32)  # exact: r has 8 significant bits
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------
# layer-ahead query prediction  (section 3.3, Algorithm 1, query-prediction step)
# ---------------------------------------------------------------------------
def predict_q(X_bits, W_bits) -> np.ndarray:
    """Q_pred = X W_Q^T in fp64.

    X is [M][K] (one row per sequence: the layer input X^i), W_Q is [N][K] in
    the usual linear-layer layout (N = Hq * D output features).  The page
    writes W_Q^{i+1} X^i with column vectors; with row vectors that is X W^T.
    """
    X = bf16_to_f64(X_bits)
    W = bf16_to_f64(W_bits)
    return X @ W.T


# ---------------------------------------------------------------------------
# block digests  (section 2.2: Quest min/max pooling, MoBA mean pooling)
# ---------------------------------------------------------------------------
def valid_tokens(j: int, P: int, seq_len: int) -> np.ndarray:
    """Token positions of block j that exist: [jP, min((j+1)P, seq_len))."""
    return np.arange(j * P, min((j + 1) * P, seq_len))


def digest_minmax(K_bits, seq_len: int, P: int):
    """Channel-wise (min, max) of K over the valid tokens of every valid block.

    K_bits: [>= nvalid*P][D] bf16 bits of one (sequence, KV head).
    Returns (mn, mx), each [nvalid][D] float64 (exact bf16 values).
    """
    K = bf16_to_f64(K_bits)
    nvalid = -(-seq_len // P)
    mn = np.empty((nvalid, K.shape[1]))
    mx = np.empty((nvalid, K.shape[1]))
    for j in range(nvalid):
        rows = K[valid_tokens(j, P, seq_len)]
        mn[j] = rows.min(axis=0)
        mx[j] = rows.max(axis=0)
    return mn, mx


def digest_mean(K_bits, seq_len: int, P: int) -> np.ndarray:
    """Channel-wise mean of K over the valid tokens of every valid block ([nvalid][D])."""
    K = bf16_to_f64(K_bits)
    nvalid = -(-seq_len // P)
    out = np.empty((nvalid, K.shape[1]))
    for j in range(nvalid):
        rows = K[valid_tokens(j, P, seq_len)]
        out[j] = rows.sum(axis=0) / rows.shape[0]
    return out


# ---------------------------------------------------------------------------
# digest scores  (section 3.2: dot product of the query with each block digest)
# ---------------------------------------------------------------------------
def scores_minmax(q_group, mn, mx) -> np.ndarray:
    """Quest upper bound u_h(j) = sum_c max(q_hc mn_jc, q_hc mx_jc); [G][nvalid]."""
    q = np.asarray(q_group, dtype=np.float64)
    a = q[:, None, :] * mn[None, :, :]
    b = q[:, None, :] * mx[None, :, :]
    return np.maximum(a, b).sum(axis=2)


def scores_mean(q_group, mean) -> np.ndarray:
    """MoBA score u_h(j) = q_h . mean_j; [G][nvalid]."""
    return np.asarray(q_group, dtype=np.float64) @ mean.T


def pool_group(u) -> np.ndarray:
    """One score per block for the KV head: the maximum over its G query heads."""
    return np.asarray(u).max(axis=0)


def pool_group_sum(u) -> np.ndarray:
    """The other pooling of a GQA group (a variant; the pages name none): the sum of the block's
    scores over the G query heads.  For the mean digest it is the group's summed query dotted
    with the digest; for the min/max bound it bounds the group's summed logit q_sum . k_t."""
    return np.asarray(u).sum(axis=0)


# ---------------------------------------------------------------------------
# top-k selection and residency split  (section 3.3, Algorithm 1: B_pred, B_cpu)
# ---------------------------------------------------------------------------
def select_topk(U, k: int) -> np.ndarray:
    """B_pred: the k_eff = min(k, len(U)) best blocks by (score desc, index asc).

    Returned in ascending block order.
    """
    U = np.asarray(U, dtype=np.float64)
    n = U.shape[0]
    order = sorted(range(n), key=lambda j: (-U[j], j))
    return np.array(sorted(order[: min(k, n)]), dtype=np.int64)


def split_residency(selected, resident_mask):
    """(S intersect R, S minus R) in ascending order; the second is B_cpu."""
    res = [int(j) for j in selected if resident_mask[j]]
    cpu = [int(j) for j in selected if not resident_mask[j]]
    return np.array(res, dtype=np.int64), np.array(cpu, dtype=np.int64)


def delta_list(cpu, prev_cpu) -> np.ndarray:
    """Blocks of the new CPU list that were not in the previous one (ascending)."""
    prev = set(int(j) for j in prev_cpu)
    return np.array([int(j) for j in cpu if int(j) not in prev], dtype=np.int64)


# ---------------------------------------------------------------------------
# asynchronous periodic recall  (section 3.4)
# ---------------------------------------------------------------------------
def recall_plan(U, selected, resident_mask, slot_of):
    """One unit's recall at a recall step (section 3.4: important blocks are copied back
    into GPU memory).  Reading of the policy, which the pages leave open:

    * the blocks brought in are the selected blocks that are not resident, the most
      important first (score descending, lower index first);
    * each takes the pool slot of a resident block that is not selected, the least
      important first (score ascending, lower index first), so the resident set keeps its
      size;
    * the recall stops when either side runs out.

    U: scores per block (all blocks of the unit's table); selected: the top-k blocks;
    resident_mask: bool per block; slot_of: pool slot per block.  Returns the ops
    (block, slot, evicted block) in ascending order of the block brought in.
    """
    U = np.asarray(U, dtype=np.float64)
    sel = set(int(j) for j in selected)
    incoming = sorted((int(j) for j in sel if not resident_mask[j]), key=lambda j: (-U[j], j))
    evictable = sorted((j for j in range(len(resident_mask)) if resident_mask[j] and j not in sel),
                       key=lambda j: (U[j], j))
    n = min(len(incoming), len(evictable))
    ops = [(incoming[i], int(slot_of[evictable[i]]), evictable[i]) for i in range(n)]
    return sorted(ops)


def apply_recall(slot_of, resident_mask, ops):
    """Page-table and residency of the unit after its recall ops: evictions first, then
    the recalled blocks take their slots."""
    slot_of = np.array(slot_of, copy=True)
    resident_mask = np.array(resident_mask, dtype=bool, copy=True)
    for _, _, e in ops:
        slot_of[e] = -1
        resident_mask[e] = False
    for b, slot, _ in ops:
        slot_of[b] = slot
        resident_mask[b] = True
    return slot_of, resident_mask


def recall_plan_pages(U_heads, selected_heads, resident_mask, slot_of_heads):
    """One sequence's recall with residency per page, a page being one block for all KV heads
    (the 128 KB transfer unit of the pages' PCIe comparison; section 3.4 for the recall).
    Reading, which the pages leave open: the pages some head selects that are not resident come
    in, the most important first, importance being the largest of the heads' scores (ties to the
    lower block); each replaces a resident page that no head selects, the least important first;
    the plan stops when either side runs out.  U_heads [Hkv][nblk] pooled scores,
    selected_heads: each head's selected blocks, resident_mask [nblk] (the sequence's pages),
    slot_of_heads [Hkv][nblk].  Returns, per head, [(block in, its slot, block out)] in
    ascending block-in order."""
    Hkv, nblk = len(U_heads), len(resident_mask)
    importance = [max(float(U_heads[h][j]) for h in range(Hkv)) for j in range(nblk)]
    chosen = set()
    for blocks in selected_heads:
        chosen.update(int(j) for j in blocks)
    need = sorted((j for j in chosen if not resident_mask[j]), key=lambda j: (-importance[j], j))
    free = sorted((j for j in range(nblk) if resident_mask[j] and j not in chosen), key=lambda j: (importance[j], j))
    pairs = sorted(zip(need, free))
    return [[(j_in, int(slot_of_heads[h][j_out]), j_out) for j_in, j_out in pairs] for h in range(Hkv)]


def recall_intervals(traces, beta=0.12):
    """Per-layer recall intervals from an offline profile (section 3.4: for each layer, the
    largest number of steps that keeps the measured CPU compute ratio below the threshold beta,
    12% by default).  traces[l][s] is layer l's ratio at the (s+1)-th step after a refresh.
    Readings: every step of the interval must be below beta (strictly); an interval is at least
    one step (recall every step) and at most the profiled length."""
    out = []
    for trace in traces:
        best = 0
        for n in range(1, len(trace) + 1):  # every candidate length, checked in full
            if all(float(r) < beta for r in trace[:n]):
                best = n
        out.append(max(best, 1))
    return out


# ---------------------------------------------------------------------------
# partial attention and merge  (section 3.2; FlashAttention / online softmax)
# ---------------------------------------------------------------------------
def block_tokens(blocks, P: int, seq_len: int) -> np.ndarray:
    if len(blocks) == 0:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([valid_tokens(int(j), P, seq_len) for j in blocks]).astype(np.int64)


def attention_partial(q, K, V, scale: float):
    """Softmax attention of one query over a token set.

    q [D], K [n][D], V [n][D] float64.  Returns (O [D] normalised, LSE) with
    LSE = ln sum_t exp(scale * q.k_t); the empty set gives (0, -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(q.shape[0]), NEG_INF
    s = scale * (K @ q)
    m = s.max()
    w = np.exp(s - m)
    l = w.sum()
    return (w @ V) / l, m + math.log(l)


def merge(O1, L1, O2, L2):
    """Combine two normalised partials by their log-sum-exp weights.

    O = (e^L1 O1 + e^L2 O2) / (e^L1 + e^L2), L = ln(e^L1 + e^L2), evaluated with
    the larger LSE factored out; two empty partials give (0, -inf).
    """
    O1 = np.asarray(O1, dtype=np.float64)
    O2 = np.asarray(O2, dtype=np.float64)
    m = max(L1, L2)
    if m == NEG_INF:
        return np.zeros_like(O1), NEG_INF
    w1 = math.exp(L1 - m)
    w2 = math.exp(L2 - m)
    return (w1 * O1 + w2 * O2) / (w1 + w2), m + math.log(w1 + w2)


# ---------------------------------------------------------------------------
# one (sequence, KV head): the whole step  (Algorithm 1, one layer)
# ---------------------------------------------------------------------------
def unit_step(q_sel_bits, q_attn_bits, K_bits, V_bits, seq_len: int, P: int, k: int, kind: str,
              resident_mask, scale: float, prev_cpu=None, pool: str = "max", gpu_blocks: str = "selected"):
    """Selection with q_sel (the predicted query), GPU partial with q_attn.

    q_sel_bits, q_attn_bits: [G][D] bf16 bits of the group's query heads.
    Returns a dict with scores (pooled, [nvalid]), per-head scores, topk, res,
    cpu, delta, and per-head GPU partials (O [G][D], L [G]) over the blocks the GPU
    attends: S intersect R (``gpu_blocks="selected"``, the reading of section 3.2), or
    every valid resident block R (``"resident"``, the other reading of Algorithm 1's
    GPUATTN(Q, B_gpu), a variant; its merge with the CPU partial over S minus R is then
    attention over R union S).  ``pool``: "max" (default) or "sum" over the group.
    """
    qs = bf16_to_f64(q_sel_bits)
    qa = bf16_to_f64(q_attn_bits)
    if kind == "minmax":
        mn, mx = digest_minmax(K_bits, seq_len, P)
        u = scores_minmax(qs, mn, mx)
    elif kind == "mean":
        u = scores_mean(qs, digest_mean(K_bits, seq_len, P))
    else:
        raise ValueError(kind)
    if pool not in ("max", "sum"):
        raise ValueError(pool)
    U = (pool_group(u) if pool == "max" else pool_group_sum(u)) if u.shape[1] else np.zeros(0)
    S = select_topk(U, k)
    res, cpu = split_residency(S, resident_mask)
    delta = delta_list(cpu, prev_cpu if prev_cpu is not None else [])
    K = bf16_to_f64(K_bits)
    V = bf16_to_f64(V_bits)
    if gpu_blocks == "selected":
        gpu = res
    elif gpu_blocks == "resident":
        nvalid = -(-seq_len // P)
        gpu = np.flatnonzero(np.asarray(resident_mask, dtype=bool)[:nvalid])
    else:
        raise ValueError(gpu_blocks)
    toks = block_tokens(gpu, P, seq_len)
    G = qa.shape[0]
    O = np.zeros((G, qa.shape[1]))
    L = np.full(G, NEG_INF)
    for h in range(G):
        O[h], L[h] = attention_partial(qa[h], K[toks], V[toks], scale)
    return dict(scores=U, head_scores=u, topk=S, res=res, cpu=cpu, delta=delta, gpu=gpu, O=O, L=L)
