// scout_sparse_attn: split-K paged GQA decode attention over the resident
// selected blocks.  ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1
// (A_gpu = GPUATTN(Q, B_gpu)): the GPU attends the top-k blocks in its memory.
//
// Work partition (balanced over the SMs): the resident selected blocks of all
// units form one list of N = sum_u res_count[u] blocks.  CTA c of Gp = min(grid,
// N) takes the contiguous range [c N / Gp, (c+1) N / Gp).  A unit that falls
// inside one range is finished by that CTA; a unit split over several CTAs is
// finished by the last of them to arrive (self-resetting counter), which merges
// the per-CTA partials by their LSE.  Only a range's first and last segment can be
// cut, and the range is walked last segment first: both of a CTA's cut pieces are
// then produced early, and a dedicated split warp counts them and does the
// cross-CTA merge (dependent global round trips) while the whole units stream.
// When the grid covers every unit and no unit is large (at most kUnitSubPagesPerWarp
// sub-pages per consumer warp), CTA c takes unit c whole instead: nothing is cut, so
// no cross-CTA merge (round trips that wait behind the K/V copies in flight) ends
// the launch, and the longest CTA has one unit's pages.
//
// Inside a CTA: the NC consumer warps (six, or four when a larger group's combine
// state needs the room) take the range's sub-pages round-robin.  Each warp owns
// kStages / NC stages of a shared-memory ring and keeps them filled itself: when
// it has finished a sub-page it reloads that stage with its sub-page kStages / NC
// further on (one 3-D TMA box per K and per V sub-page,
// 128-byte swizzle, completion on an mbarrier), so a stage is never idle while
// another warp is behind.  The lanes resolve the warp's next 32 sub-pages (list
// entry, page-table slot, valid tokens) one batch ahead, so the dependent
// global loads stay off the critical path.  Per sub-page a warp runs S = Q K^T
// and O += P V on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate;
// P is split into a bf16 high and low part so the probabilities keep ~16
// significant bits) and keeps an online softmax, combined through shared memory
// at the end of each unit segment by the epilogue warp.
#include "common.cuh"

namespace scout {
namespace {

// Consumer warps and tokens per stage: six warps with 32-token stages, two per warp in a 192 KB
// ring.  The warps are latency-bound (each page is a chain of ldmatrix, MMA and softmax steps),
// so more of them per scheduler hide more of it.  Measured on GB300, Qwen3-14B-shaped step
// (graph replay, same box, back to back): four warps (three stages each) 58.36 us per step and
// 33.3 us alone, six 57.78 us and 30.1 us alone, six with two pages per pass 59.08 us; eight
// warps with 16-token stages were ~15% slower than four (the per-page overhead doubles).  Six
// warps' combine state leaves room for the whole ring and two combine slots up to G = 5 at 320
// units (with one slot, warps that finish a short segment wait for the epilogue to drain the
// previous one); past that a launch takes one slot, then four warps (three stages each, a
// smaller combine state), then a smaller ring.
#ifndef SCOUT_ATTN_CONSUMERS
#define SCOUT_ATTN_CONSUMERS 6
#endif
constexpr int kFallbackConsumers = 4;
#ifndef SCOUT_ATTN_SUBPAGE
#define SCOUT_ATTN_SUBPAGE 32
#endif
#ifndef SCOUT_ATTN_PAIR
#define SCOUT_ATTN_PAIR 1
#endif

constexpr int kConsumers = SCOUT_ATTN_CONSUMERS;  // the preferred count; the kernel takes it as NC
constexpr int kSubTokens = SCOUT_ATTN_SUBPAGE;
// pages a consumer warp attends in one pass (1 or 2); measured on GB300 in the graph-replayed
// Qwen3-14B-shaped step: one 59.55 us per step, two 60.35 (with one, a stage holds a page for
// less time, so more of the ring is loading)
constexpr int kPair = SCOUT_ATTN_PAIR;

// warps of a CTA with NC consumer warps: the consumers, then an epilogue warp (combines the
// warps' states, writes whole units) and a split warp (merges the units cut by range boundaries)
template <int NC>
__host__ __device__ constexpr int threads_of() { return (NC + 2) * 32; }
constexpr int kMaxSplit = 2;  // pieces of cut units per CTA range: its first and its last segment
constexpr int kPhaseB = 8;   // page of a batch at which the next batch's page-table loads are issued
constexpr int kPhaseC = 16;  // and at which their values are used
// A launch whose grid covers every unit gives each CTA one whole unit when no unit has more than
// this many sub-pages per consumer warp; otherwise the flattened blocks are split evenly.
constexpr int kUnitSubPagesPerWarp = 8;
constexpr int kMaxUnits = 4096;
// resident-list entries (units x k) a launch may address: the prefix over the counts and the
// per-range sub-page numbers (up to two sub-pages per block) then fit a 32-bit int
constexpr int64_t kMaxEntries = (int64_t)1 << 28;
constexpr int kMaxSlots = 2;  // combine slots between the consumer warps and the epilogue warp
constexpr int kMaxGrid = 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// A stage holds K and V of one sub-page of PS tokens (a block streams as P / PS
// sub-pages); the ring has S stages and every consumer warp owns kPerWarp of them.
constexpr int kRingTarget = 192 * 1024;
template <int P, int NC>
constexpr int big_ring() {  // stages of the 192 KB ring
  return kRingTarget / (4 * (P < kSubTokens ? P : kSubTokens) * 128) / NC * NC;
}
template <int P, int NC>
constexpr int small_ring() {  // two thirds of it, for groups and batches whose combine state is large
  return big_ring<P, NC>() * 2 / 3 / NC * NC;
}
template <int P, int S, int NC>
struct Cfg {
  static constexpr int PS = P < kSubTokens ? P : kSubTokens;  // tokens per stage
  static constexpr int kSub = P / PS;                          // stages per block
  static constexpr int kStages = S;
  static constexpr int kPerWarp = kStages / NC;
  static constexpr int kHalfBytes = PS * 128;        // one 64-column half of a sub-page
  static constexpr int kStageBytes = 4 * kHalfBytes; // K (2 halves) + V (2 halves)
  static constexpr int kRingBytes = kStages * kStageBytes;
  static_assert(kStages % NC == 0 && kPhaseB < kPhaseC && kPhaseC < 32 - kPerWarp - 1,
                "stage ownership and resolution phases");

};

struct AttnArgs {
  const __nv_bfloat16* q;
  const int32_t* page_table;
  const int32_t* seq_len;
  const int32_t* res_list;
  const int32_t* res_count;
  int Hq, Hkv, G, nblk_cap, k, units;
  int64_t n_slots;
  float scale_log2;  // scale * log2(e)
  int nslots;  // combine slots that fit in shared memory (1 or 2)
  float* O_part;
  float* lse_part;
  // merge mode (O_out != nullptr): the CPU partial is merged in and bf16 O written
  const float* O_cpu;
  const float* lse_cpu;
  __nv_bfloat16* O_out;
  float* lse_out;
  int32_t* counters;   // [units]
  float* slot_lse;     // [kMaxGrid][2][kMaxG]
  float* slot_O;       // [kMaxGrid][2][kMaxG][kD]
  int32_t* status;
};

// first CTA whose range contains flattened position x (all Gp ranges non-empty)
__device__ __forceinline__ int cta_of(int64_t x, int64_t N, int Gp) {
  return (int)(((x + 1) * Gp + N - 1) / N) - 1;
}
__device__ __forceinline__ int64_t range_start(int c, int64_t N, int Gp) { return (int64_t)c * N / Gp; }

// Row address (shared::cta) of token r, 16-byte chunk C (dims 8C..8C+7) in a sub-page
// of PS tokens stored as two 64-column halves with the 128-byte TMA swizzle.
template <int PS>
__device__ __forceinline__ uint32_t page_addr(uint32_t base, int r, int C) {
  return base + (uint32_t)((C >> 3) * PS * 128 + r * 128 + ((((C & 7) ^ (r & 7))) << 4));
}

// Zero the V rows of tokens ntok .. PS-1 of a stage (the part of a sequence's last page
// past its end), so that their zero probabilities never meet non-finite stale values.
template <int PS>
__device__ __forceinline__ void clear_tail_rows(uint8_t* vstage, int ntok, int lane) {
  // two 64-column halves of PS rows x 128 bytes; 8 lanes per 128-byte row
  for (int idx = ntok * 8 + lane; idx < PS * 8; idx += 32) {
    const int r = idx >> 3, c = idx & 7;
    *reinterpret_cast<uint4*>(vstage + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(vstage + PS * 128 + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
  }
  __syncwarp();
}

struct WarpState {
  float m[2];  // running max of scaled scores (log2 units) of heads 2t, 2t+1
  float l[2];  // running sum of exp2(s - m) over this lane's tokens, heads 2t, 2t+1
  float o[8][4];  // O^T accumulators: dims 16md + g (+8) x heads 2t, 2t+1
};

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// NP pages of one warp at once, computed transposed so that tokens and head dims fill the
// MMA's M:
//   S^T = K Q^T (tokens x heads), online softmax per head (column),
//   O^T += V^T P^T (dims x heads); P^T reaches the B-operand layout by movmatrix.
// Taking two pages together gives the MMA chains of both to the scheduler at once and
// pays the running-max rescale once.  qb holds Q^T fragments: qb[s] = heads g, dims
// 16s + 2t (+8).  The work is cut in two, so that the K halves of the stages can be refilled
// as soon as the scores are computed, while the softmax and P V still run:
//   attend_scores   s = scale * log2(e) * K q (masked past ntok), reading only K;
//   attend_values   the online-softmax update and O^T += V^T P^T, reading only V.
template <int PS, int NP>
__device__ __forceinline__ void attend_scores(const uint32_t (&kbase)[NP], const int (&ntok)[NP],
                                              const uint32_t (&qb)[8][2], float scale_log2,
                                              float (&s)[NP * (PS / 16)][4], int lane) {
  constexpr int MT = PS / 16;  // 16-token tiles per stage
  constexpr int T = NP * MT;   // tiles in all
  const int g = lane >> 2;
#pragma unroll
  for (int tt = 0; tt < T; ++tt) {
    const int pg = tt / MT, mt = tt % MT;
    float s2[4] = {0.f, 0.f, 0.f, 0.f};  // second accumulator: halves the dependent MMA chain
    s[tt][0] = s[tt][1] = s[tt][2] = s[tt][3] = 0.f;
    const int r = mt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
    for (int ks = 0; ks < 8; ks += 2) {
      uint32_t a0, a1, a2, a3, c0, c1, c2, c3;
      ldsm_x4(page_addr<PS>(kbase[pg], r, 2 * ks + (lane >> 4)), a0, a1, a2, a3);
      ldsm_x4(page_addr<PS>(kbase[pg], r, 2 * ks + 2 + (lane >> 4)), c0, c1, c2, c3);
      mma_bf16(s[tt], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
      mma_bf16(s2, c0, c1, c2, c3, qb[ks + 1][0], qb[ks + 1][1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) s[tt][e] += s2[e];
  }
#pragma unroll
  for (int tt = 0; tt < T; ++tt) {
    const int pg = tt / MT, mt = tt % MT;
    const int t0 = mt * 16 + g, t1 = t0 + 8;
    s[tt][0] = t0 < ntok[pg] ? s[tt][0] * scale_log2 : -INFINITY;
    s[tt][1] = t0 < ntok[pg] ? s[tt][1] * scale_log2 : -INFINITY;
    s[tt][2] = t1 < ntok[pg] ? s[tt][2] * scale_log2 : -INFINITY;
    s[tt][3] = t1 < ntok[pg] ? s[tt][3] * scale_log2 : -INFINITY;
  }
}

template <int PS, int NP>
__device__ __forceinline__ void attend_values(const uint32_t (&vbase)[NP], float (&s)[NP * (PS / 16)][4],
                                              WarpState& st, int lane) {
  constexpr int MT = PS / 16;
  constexpr int T = NP * MT;
  // per-head (column) max over the pages' tokens
  float bm0 = -INFINITY, bm1 = -INFINITY;
#pragma unroll
  for (int tt = 0; tt < T; ++tt) {
    bm0 = fmaxf(bm0, fmaxf(s[tt][0], s[tt][2]));
    bm1 = fmaxf(bm1, fmaxf(s[tt][1], s[tt][3]));
  }
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o));
    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o));
  }
  const float n0 = fmaxf(st.m[0], bm0), n1 = fmaxf(st.m[1], bm1);
  const float al0 = exp2f(st.m[0] - n0), al1 = exp2f(st.m[1] - n1);  // 0 on the first pages
  st.m[0] = n0;
  st.m[1] = n1;
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int tt = 0; tt < T; ++tt) {
    s[tt][0] = exp2f(s[tt][0] - n0);
    s[tt][1] = exp2f(s[tt][1] - n1);
    s[tt][2] = exp2f(s[tt][2] - n0);
    s[tt][3] = exp2f(s[tt][3] - n1);
    ps0 += s[tt][0] + s[tt][2];
    ps1 += s[tt][1] + s[tt][3];
  }
  st.l[0] = st.l[0] * al0 + ps0;
  st.l[1] = st.l[1] * al1 + ps1;
  // the running sums move only when some head's maximum rose (rarely, after the first pages)
  if (!__all_sync(0xffffffffu, al0 == 1.f && al1 == 1.f)) {
#pragma unroll
    for (int md = 0; md < 8; ++md) {
      st.o[md][0] *= al0;
      st.o[md][1] *= al1;
      st.o[md][2] *= al0;
      st.o[md][3] *= al1;
    }
  }
#pragma unroll
  for (int tt = 0; tt < T; ++tt) {
    const int pg = tt / MT, mt = tt % MT;
    // P^T as B operand (k = tokens, n = heads), split into bf16 high and low parts
    const uint32_t ht = pack_bf16(s[tt][0], s[tt][1]), hb = pack_bf16(s[tt][2], s[tt][3]);
    const uint32_t lt = pack_bf16(s[tt][0] - bf16_lo(ht), s[tt][1] - bf16_hi(ht));
    const uint32_t lb = pack_bf16(s[tt][2] - bf16_lo(hb), s[tt][3] - bf16_hi(hb));
    const uint32_t bh0 = movmatrix_t(ht), bh1 = movmatrix_t(hb);
    const uint32_t bl0 = movmatrix_t(lt), bl1 = movmatrix_t(lb);
    const int r = mt * 16 + (lane >> 4) * 8 + (lane & 7);
#pragma unroll
    for (int md = 0; md < 8; ++md) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4_t(page_addr<PS>(vbase[pg], r, 2 * md + ((lane >> 3) & 1)), a0, a1, a2, a3);
      mma_bf16(st.o[md], a0, a1, a2, a3, bh0, bh1);
      mma_bf16(st.o[md], a0, a1, a2, a3, bl0, bl1);
    }
  }
}

// One segment's per-warp softmax states, handed from the consumer warps to the
// epilogue warp through shared memory.  A slot holds m[warps][8], l[warps][8] and
// O^T partials o[warps][G][128] (fp32); its size depends on G.
__host__ __device__ constexpr int slot_floats(int G, int NC) { return 2 * NC * kMaxG + NC * G * kD; }
template <int NC>
struct SlotView {
  float* base;
  int G;
  __device__ float& m(int w, int h) const { return base[w * kMaxG + h]; }
  __device__ float& l(int w, int h) const { return base[(NC + w) * kMaxG + h]; }
  __device__ float* o(int w, int h) const { return base + 2 * NC * kMaxG + (w * G + h) * kD; }
};

// Walks the unit segments of one CTA's flattened block range in processing order: the
// range's last segment first (when the range holds more than one), then the others from the
// start.  The last and the first segment are the ones a range boundary can cut, so both of
// a CTA's pieces of units shared with its neighbours come early, and the cross-CTA merge of
// those units (dependent global round trips) overlaps the streaming of the whole units.
struct SegIter {
  const int* prefix;
  int64_t pos, end;  // the in-order walk over [start, end of the walk)
  int u;
  bool rot;          // the rotated-in last segment is still to come
  int rot_u;
  int64_t rot_lo, rot_hi;
  __device__ __forceinline__ bool next(int& uu, int64_t& lo, int64_t& hi) {
    if (rot) {
      rot = false;
      uu = rot_u;
      lo = rot_lo;
      hi = rot_hi;
      return true;
    }
    while (pos < end) {
      const int64_t h = min(end, (int64_t)prefix[u + 1]);
      if (h > pos) {
        uu = u;
        lo = pos;
        hi = h;
        pos = h;
        ++u;
        return true;
      }
      ++u;
    }
    return false;
  }
};

__device__ __forceinline__ int unit_of(const int* prefix, int units, int64_t x, int lo = 0) {
  int hi = units - 1;  // last unit with prefix[u] <= x: the unit holding x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The processing order of a CTA's range [start, end): its last unit segment [last_lo, end)
// first, then [start, last_lo).  at(p) is the block at position p of that order.
struct RangeOrder {
  int64_t start, end, last_lo;
  __device__ __forceinline__ int64_t at(int64_t p) const {
    const int64_t nl = end - last_lo;
    return p < nl ? last_lo + p : start + (p - nl);
  }
};
__device__ __forceinline__ RangeOrder range_order(const int* prefix, int units, int64_t start, int64_t end) {
  int64_t last_lo = start;
  if (end > start) last_lo = max(start, (int64_t)prefix[unit_of(prefix, units, end - 1)]);
  return RangeOrder{start, end, last_lo};
}
__device__ __forceinline__ SegIter seg_iter(const int* prefix, int units, const RangeOrder& ro) {
  const bool rot = ro.last_lo > ro.start;  // more than one segment: the last one goes first
  const int u_last = ro.end > ro.start ? unit_of(prefix, units, ro.end - 1) : 0;
  return SegIter{prefix, ro.start, rot ? ro.last_lo : ro.end, unit_of(prefix, units, ro.start), rot, u_last,
                 ro.last_lo, ro.end};
}

// Q^T fragments (B operand) of unit u: head g, dims 16 ks + 2t (+8); zero for g >= G.
__device__ __forceinline__ void load_q(const AttnArgs& a, int u, int lane, uint32_t (&qf)[8][2]) {
  const int g = lane >> 2, t = lane & 3;
  const int b = u / a.Hkv, kvh = u - b * a.Hkv;
  const __nv_bfloat16* qrow = a.q + ((int64_t)b * a.Hq + (int64_t)kvh * a.G + g) * kD;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    qf[ks][0] = g < a.G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * t) : 0u;
    qf[ks][1] = g < a.G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * t) : 0u;
  }
}

// The CPU partial of a unit (merge only): lane l holds dims 4l .. 4l+3 of every head and the
// LSE of head l.  Loaded ahead of its use so that the latency overlaps other work.
struct CpuPart {
  float4 o[kMaxG];
  float lse;
};
__device__ __forceinline__ void load_cpu(const AttnArgs& a, int uu, int lane, CpuPart& cp) {
  if (a.O_out == nullptr) return;
#pragma unroll
  for (int h = 0; h < kMaxG; ++h)
    if (h < a.G) cp.o[h] = __ldcs(reinterpret_cast<const float4*>(a.O_cpu + ((int64_t)uu * a.G + h) * kD + 4 * lane));
  cp.lse = lane < a.G ? __ldcs(a.lse_cpu + (int64_t)uu * a.G + lane) : -INFINITY;
}
// The final per-head GPU LSE of unit uu is in fin[]: write it (partial), or its merge with the
// CPU partial, leaving the merge weights in wg[] / wc[] (one warp; per-warp shared scratch).
__device__ __forceinline__ void unit_final(const AttnArgs& a, int uu, int lane, const float* fin, float* wgs,
                                           float* wcs, const CpuPart& cp) {
  if (lane < a.G) {
    const int64_t r = (int64_t)uu * a.G + lane;
    const float lg = fin[lane];
    if (a.O_out != nullptr) {
      const float lc = cp.lse, m = fmaxf(lg, lc);
      float wg = 0.f, wc = 0.f, lse = -INFINITY;
      if (m != -INFINITY) {
        wg = expf(lg - m);
        wc = expf(lc - m);
        const float sum = wg + wc;
        lse = m + logf(sum);
        wg /= sum;
        wc /= sum;
      }
      wgs[lane] = wg;
      wcs[lane] = wc;
      if (a.lse_out != nullptr) a.lse_out[r] = lse;
    } else {
      a.lse_part[r] = lg;
    }
  }
  __syncwarp();
}
// Dims 4 lane .. 4 lane + 3 of head h of unit uu: the GPU partial o, or its merge with the CPU
// partial by the weights unit_final left.
__device__ __forceinline__ void store4(const AttnArgs& a, int uu, int h, int lane, float4 o, const float* wgs,
                                       const float* wcs, const CpuPart& cpu) {
  const int64_t off = ((int64_t)uu * a.G + h) * kD + 4 * lane;
  if (a.O_out != nullptr) {
    const float4 cp = cpu.o[h];
    const float wg = wgs[h], wc = wcs[h];
    uint2 pk;
    pk.x = pack_bf16(wg * o.x + wc * cp.x, wg * o.y + wc * cp.y);
    pk.y = pack_bf16(wg * o.z + wc * cp.z, wg * o.w + wc * cp.w);
    *reinterpret_cast<uint2*>(a.O_out + off) = pk;
  } else {
    *reinterpret_cast<float4*>(a.O_part + off) = o;
  }
}

// The split warp of a CTA: a unit cut by range boundaries has one piece per CTA range it
// touches (c0 .. c1).  Each piece is stored to its workspace slot by the CTA's epilogue warp,
// which signals it on sbar; the split warp counts it, and the piece that completes the count
// (last to arrive) merges all of them by their LSE.  Nothing waits on another CTA.
__device__ void run_split_warp(const AttnArgs& a, const int* prefix, int64_t N, int Gp, int c, uint64_t* sbar,
                               float* sfin, float* swg, float* swc, int lane) {
  const int64_t start = range_start(c, N, Gp), end = range_start(c + 1, N, Gp);
  SegIter it = seg_iter(prefix, a.units, range_order(prefix, a.units, start, end));
  int u, k = 0;
  int64_t lo, hi;
  CpuPart cpu;
  while (it.next(u, lo, hi)) {
    if (lo == prefix[u] && hi == prefix[u + 1]) continue;  // whole: the epilogue warp's
    if (k >= kMaxSplit) break;  // a range has at most two cut segments
    load_cpu(a, u, lane, cpu);  // used only if this piece completes the unit
    // the epilogue's stores of the piece happen before its arrive; the fence below makes them
    // visible, with this warp's, to the CTA that merges the unit
    if (!mbar_wait(&sbar[k], 0u) && lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
    ++k;
    const int c0 = cta_of(prefix[u], N, Gp), c1 = cta_of(prefix[u + 1] - 1, N, Gp);
    auto piece_slot = [&](int cc) {
      return (int64_t)cc * 2 + (prefix[u] <= range_start(cc, N, Gp) ? 0 : 1);
    };
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(&a.counters[u], 1) == c1 - c0;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) continue;
    __threadfence();
    // merge the pieces by their LSE in one pass (running max per head): every load of a
    // piece is issued at once
    float mx[kMaxG], sm[kMaxG];
    float4 acc[kMaxG];
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
      mx[h] = -INFINITY;
      sm[h] = 0.f;
      acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int cc = c0; cc <= c1; ++cc) {
      float pl[kMaxG];
      float4 po[kMaxG];
      const int64_t sl = piece_slot(cc);
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h >= a.G) continue;
        pl[h] = __ldcg(a.slot_lse + sl * kMaxG + h);
        po[h] = __ldcg(reinterpret_cast<const float4*>(a.slot_O + (sl * kMaxG + h) * kD + 4 * lane));
      }
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) {
        if (h >= a.G || pl[h] == -INFINITY) continue;  // a piece without tokens weighs nothing
        const float nm = fmaxf(mx[h], pl[h]);
        const float keep = mx[h] == -INFINITY ? 0.f : expf(mx[h] - nm), w = expf(pl[h] - nm);
        acc[h].x = acc[h].x * keep + w * po[h].x;
        acc[h].y = acc[h].y * keep + w * po[h].y;
        acc[h].z = acc[h].z * keep + w * po[h].z;
        acc[h].w = acc[h].w * keep + w * po[h].w;
        sm[h] = sm[h] * keep + w;
        mx[h] = nm;
      }
    }
    float fin = -INFINITY;
#pragma unroll
    for (int h = 0; h < kMaxG; ++h)
      if (h == lane && sm[h] > 0.f) fin = mx[h] + logf(sm[h]);
    if (lane < a.G) sfin[lane] = fin;
    __syncwarp();
    unit_final(a, u, lane, sfin, swg, swc, cpu);
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
      if (h >= a.G) continue;
      const float r = sm[h] > 0.f ? 1.f / sm[h] : 0.f;
      store4(a, u, h, lane, make_float4(acc[h].x * r, acc[h].y * r, acc[h].z * r, acc[h].w * r), swg, swc, cpu);
    }
    __syncwarp();
    if (lane == 0) a.counters[u] = 0;  // ready for the next call
  }
}

// UNITS: the launch's grid covers every unit, so the whole-unit partition may be taken (the
// other instance compiles the flattened split alone).
template <int P, int S, int NC, bool UNITS>
__global__ void __launch_bounds__(threads_of<NC>(), 1) sparse_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV,
                                                                  const AttnArgs a) {
  using C = Cfg<P, S, NC>;
  constexpr int kConsumerWarps = NC, kEpilogueWarp = NC, kSplitWarp = NC + 1, kThreads = threads_of<NC>();
  extern __shared__ uint8_t smem_raw[];
  // kfull / vfull: the K / V half of a stage has landed (one phase per fill of the stage)
  __shared__ uint64_t kfull[C::kStages], vfull[C::kStages], cfull[kMaxSlots], cempty[kMaxSlots], sbar[kMaxSplit];
  __shared__ int wtot[kThreads / 32], wmax[kThreads / 32];
  __shared__ float ew[kMaxG][kConsumerWarps], eown[kMaxG];  // epilogue weights
  __shared__ float efin[kMaxG], fwg[kMaxG], fwc[kMaxG];     // epilogue final LSE, merge weights
  __shared__ float sfin[kMaxG], swg[kMaxG], swc[kMaxG];    // split warp final LSE, merge weights

  // dynamic shared memory: [ring (1024-aligned)][combine slots][unit prefix]
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  float* cbf = reinterpret_cast<float*>(ring + C::kRingBytes);
  const int slot_f = slot_floats(a.G, NC);
  int* prefix = reinterpret_cast<int*>(cbf + a.nslots * slot_f);  // [units + 1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&vfull[i], 1);
    }
    for (int i = 0; i < a.nslots; ++i) {
      mbar_init(&cfull[i], kConsumerWarps);
      mbar_init(&cempty[i], 1);
    }
    for (int i = 0; i < kMaxSplit; ++i) mbar_init(&sbar[i], 1);
    fence_mbar_init();
  }
  if (tid == 32) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  // started early: the lists (and possibly anything else read below) are written by the kernel
  // this launch depends on; a no-op otherwise
  wait_prerequisites();
  // exclusive prefix of the clamped resident counts over all units
  {
    const int per = (a.units + kThreads - 1) / kThreads;
    const int lo = min(a.units, tid * per), hi = min(a.units, lo + per);
    int sum = 0, mx = 0;
    for (int u = lo; u < hi; ++u) {  // the counts are read once, kept in place of the prefix
      prefix[u] = min(max(a.res_count[u], 0), a.k);
      sum += prefix[u];
      if constexpr (UNITS) mx = max(mx, prefix[u]);
    }
    if constexpr (UNITS) {
      mx = __reduce_max_sync(0xffffffffu, mx);
      if (lane == 0) wmax[warp] = mx;
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += x;
    }
    if (lane == 31) wtot[warp] = inc;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += wtot[w];
    int run = base + inc - sum;
    for (int u = lo; u < hi; ++u) {
      const int n = prefix[u];
      prefix[u] = run;
      run += n;
    }
    if (tid == kThreads - 1) prefix[a.units] = run;
    __syncthreads();
  }
  const int64_t N = prefix[a.units];
  // With every unit small and the grid covering them, CTA c takes unit c whole: no unit is cut,
  // so no merge of pieces across CTAs (global round trips behind the K/V copies in flight) ends
  // the launch.  Otherwise range c is [c N / Gp, (c+1) N / Gp) of the flattened blocks.
  bool by_unit = false;
  if constexpr (UNITS) {
    int maxc = 0;  // the largest clamped count
    for (int w = 0; w < kThreads / 32; ++w) maxc = max(maxc, wmax[w]);
    by_unit = a.units <= (int)gridDim.x && maxc * C::kSub <= kUnitSubPagesPerWarp * NC;
  }
  const int Gp = by_unit ? a.units : (int)min((int64_t)gridDim.x, N);
  auto rstart = [&](int cc) -> int64_t { return by_unit ? (int64_t)prefix[cc] : range_start(cc, N, Gp); };
  const int c = blockIdx.x;

  if (warp == kEpilogueWarp) {
    // ---------------- epilogue warp ------------------------------------------
    CpuPart cpu;
    // units with no resident selected block: O = 0, lse = -inf
    for (int u = c; u < a.units; u += gridDim.x) {
      if (prefix[u + 1] != prefix[u]) continue;
      load_cpu(a, u, lane, cpu);
      if (lane < a.G) efin[lane] = -INFINITY;
      __syncwarp();
      unit_final(a, u, lane, efin, fwg, fwc, cpu);
#pragma unroll
      for (int h = 0; h < kMaxG; ++h)
        if (h < a.G) store4(a, u, h, lane, make_float4(0.f, 0.f, 0.f, 0.f), fwg, fwc, cpu);
      __syncwarp();
    }
    if (c >= Gp) return;
    const int64_t start = rstart(c), end = rstart(c + 1);
    SegIter it = seg_iter(prefix, a.units, range_order(prefix, a.units, start, end));
    int u, nsplit = 0;
    int64_t lo, hi;
    for (int sg = 0; it.next(u, lo, hi); ++sg) {
      const int slot = sg % a.nslots;
      const bool whole = lo == prefix[u] && hi == prefix[u + 1];
      if (whole) load_cpu(a, u, lane, cpu);  // in flight while the unit's pages still stream
      if (!mbar_wait(&cfull[slot], (uint32_t)(sg / a.nslots) & 1u) && lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
      const SlotView<NC> cs{cbf + slot * slot_f, a.G};
      // per-head weights of the consumer warps' states (normalised) and this piece's LSE
      if (lane < a.G) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cs.m(w, lane));
        float f[kConsumerWarps], L = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          f[w] = M == -INFINITY ? 0.f : exp2f(cs.m(w, lane) - M);
          L += cs.l(w, lane) * f[w];
        }
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) ew[lane][w] = L > 0.f ? f[w] / L : 0.f;
        eown[lane] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      }
      __syncwarp();
      // this piece's normalised output, 4 dims per lane
      auto own4 = [&](int h) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float4 o = *reinterpret_cast<const float4*>(cs.o(w, h) + 4 * lane);
          const float f = ew[h][w];
          acc.x += f * o.x;
          acc.y += f * o.y;
          acc.z += f * o.z;
          acc.w += f * o.w;
        }
        return acc;
      };
      if (whole) {
        if (lane < a.G) efin[lane] = eown[lane];
        __syncwarp();
        unit_final(a, u, lane, efin, fwg, fwc, cpu);
#pragma unroll
        for (int h = 0; h < kMaxG; ++h)
          if (h < a.G) store4(a, u, h, lane, own4(h), fwg, fwc, cpu);
      } else {
        // a unit cut by a range boundary: the piece is stored to its workspace slot (the range's
        // first or last segment) and the split warp, signalled through shared memory, counts it;
        // no global round trip holds the combine slot or this warp
        const int64_t msl = (int64_t)c * 2 + (prefix[u] <= start ? 0 : 1);
        if (lane < a.G) a.slot_lse[msl * kMaxG + lane] = eown[lane];
#pragma unroll
        for (int h = 0; h < kMaxG; ++h)
          if (h < a.G) *reinterpret_cast<float4*>(a.slot_O + (msl * kMaxG + h) * kD + 4 * lane) = own4(h);
        __syncwarp();
        if (lane == 0 && nsplit < kMaxSplit) mbar_arrive(&sbar[nsplit]);
        ++nsplit;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&cempty[slot]);  // the combine slot may be refilled
    }
    return;
  }

  if (warp == kSplitWarp) {
    if (c < Gp && !by_unit) run_split_warp(a, prefix, N, Gp, c, sbar, sfin, swg, swc, lane);  // no cut unit otherwise
    return;
  }

  // ---------------- consumer warps 0 .. NC-1 ------------------------------------
  if (c >= Gp) return;
  const int g = lane >> 2, t = lane & 3;
  const int64_t start = rstart(c), end = rstart(c + 1);
  const RangeOrder order = range_order(prefix, a.units, start, end);
  // this warp's pages: sub-page i = warp + NC k of the range, k = 0 .. n_mine-1, in stage i % kStages
  // sub-page numbers within the range fit 32 bits: the host bounds units * k by 2^28
  const int n_sub = (int)(end - start) * C::kSub;
  const int n_mine = n_sub > warp ? (n_sub - 1 - warp) / kConsumerWarps + 1 : 0;
  const uint32_t ring_s = smem_u32(ring);
  // Page kk of this warp, first half of its resolution: its unit, list entry and sequence length.
  auto resolve_a = [&](int kk, int& ru, int& rj, int& rlen) {
    ru = -1;
    rj = -1;
    rlen = 0;
    if (kk < n_mine) {
      const int64_t x = order.at((warp + kConsumerWarps * kk) / C::kSub);
      ru = unit_of(prefix, a.units, x);
      rj = a.res_list[(int64_t)ru * a.k + (x - prefix[ru])];
      rlen = a.seq_len[ru / a.Hkv];
    }
  };
  // Second half: the pool row of the sub-page and its valid tokens (0 = nothing to load).  An
  // entry outside the sequence or the pool is skipped and reported.
  // Second: the page-table slot of the list entry (issued here, first used kPhaseC - kPhaseB
  // pages later, so the load's latency stays off the warp's path).
  auto resolve_b = [&](int ru, int rj, int& rsl) {
    rsl = -1;
    if (ru >= 0 && rj >= 0 && rj < a.nblk_cap) rsl = a.page_table[(int64_t)ru * a.nblk_cap + rj];
  };
  // Third: the pool row of the sub-page and its valid tokens (0 = nothing to load).  An entry
  // outside the sequence or the pool is skipped and reported.
  auto resolve_c = [&](int kk, int ru, int rj, int rlen, int sl, int& row, int& nt) {
    row = 0;
    nt = 0;
    if (ru < 0) return;
    const int h = (warp + kConsumerWarps * kk) % C::kSub;
    const int nv = rj >= 0 && rj < a.nblk_cap ? min(P, rlen - rj * P) : 0;
    if (nv <= 0 || sl < 0 || sl >= a.n_slots) {
      if (h == 0) report(a.status, SCOUT_DEV_BAD_INDEX);
      return;
    }
    nt = min(max(nv - h * C::PS, 0), C::PS);
    row = sl * P + h * C::PS;
  };
  // Load the K (which = 0) or V (which = 1) half of page kk (one lane): both 64-column halves
  // in one box.
  auto issue = [&](int kk, int row, int nt, int which) {
    const int stage = (warp + kConsumerWarps * kk) % C::kStages;
    uint64_t* bar = which ? &vfull[stage] : &kfull[stage];
    if (nt > 0) {
      uint8_t* sp = ring + stage * C::kStageBytes + which * 2 * C::kHalfBytes;
      mbar_arrive_tx(bar, 2 * C::kHalfBytes);
      tma_load_3d(sp, which ? &tmV : &tmK, 0, row, 0, bar);
    } else {
      mbar_arrive(bar);
    }
  };
  // batch b = pages 32 b .. 32 b + 31 of this warp, page 32 b + m resolved by lane m; cur_*
  // hold batch cur_b, nxt_* batch cur_b + 1 once it is resolved
  int cur_row, cur_nt, nxt_row = 0, nxt_nt = 0, pu, pj, plen, psl, cur_b = 0;
  resolve_a(lane, pu, pj, plen);
  resolve_b(pu, pj, psl);
  resolve_c(lane, pu, pj, plen, psl, cur_row, cur_nt);
  auto nt_of = [&](int kk) {
    return __shfl_sync(0xffffffffu, (kk >> 5) == cur_b ? cur_nt : nxt_nt, kk & 31);
  };
  // page kk is next in this warp's order: move to its batch when it opens one, and start
  // resolving the batch after it (list entries now, page-table slots kPhaseB pages later)
  auto advance = [&](int kk) {
    const int m = kk & 31;
    if (m == 0 && kk > 0) {
      cur_row = nxt_row;
      cur_nt = nxt_nt;
      ++cur_b;
    }
    if (m == 0) resolve_a(kk + 32 + lane, pu, pj, plen);
    if (m == kPhaseB) resolve_b(pu, pj, psl);
    if (m == kPhaseC) resolve_c(kk - kPhaseC + 32 + lane, pu, pj, plen, psl, nxt_row, nxt_nt);
  };
  // after pages kk .. kk + n - 1 (n = 1 or 2): their stages take this warp's pages kPerWarp
  // further on, the K halves once the scores are computed, the V halves after P V; lane j
  // issues the copy of page kk + j, so the two go out together.  where() gives a lane the
  // pool row and valid tokens of its page (read before the halves are issued).
  auto where = [&](int kk, int n, int& row, int& nt) {
    const int kr = kk + C::kPerWarp + (lane < n ? lane : 0);
    const int src = kr & 31;
    const int rc = __shfl_sync(0xffffffffu, cur_row, src), rn = __shfl_sync(0xffffffffu, nxt_row, src);
    const int tc = __shfl_sync(0xffffffffu, cur_nt, src), tn = __shfl_sync(0xffffffffu, nxt_nt, src);
    const bool in_cur = (kr >> 5) == cur_b;
    row = in_cur ? rc : rn;
    nt = in_cur ? tc : tn;
  };
  auto refill = [&](int kk, int n, int row, int nt, int which) {
    const int kr = kk + C::kPerWarp + (lane < n ? lane : 0);
    if (lane < n && kr < n_mine) issue(kr, row, nt, which);
  };

  for (int r = 0; r < C::kPerWarp && r < n_mine; ++r) {
    const int row = __shfl_sync(0xffffffffu, cur_row, r), nt = __shfl_sync(0xffffffffu, cur_nt, r);
    if (lane == 0) {
      issue(r, row, nt, 0);
      issue(r, row, nt, 1);
    }
  }

  SegIter it = seg_iter(prefix, a.units, order);
  int u;
  int64_t lo, hi;
  bool have = it.next(u, lo, hi);
  uint32_t qa[8][2], qn[8][2];
  if (have) load_q(a, u, lane, qa);
  int i = 0;
  bool ok = true;  // false after a bounded wait ran out
  for (int sg = 0; have; ++sg) {
    // prefetch the next segment's query while this one streams
    SegIter peek = it;
    int un;
    int64_t lo2, hi2;
    const bool have2 = peek.next(un, lo2, hi2);
    if (have2) load_q(a, un, lane, qn);
    WarpState st;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
#pragma unroll
    for (int d = 0; d < 8; ++d) st.o[d][0] = st.o[d][1] = st.o[d][2] = st.o[d][3] = 0.f;
    // this warp's sub-pages of the segment (sub-page numbers ii = warp mod NC within the range)
    const int seg_lo = i, seg_hi = i + (int)(hi - lo) * C::kSub;
    for (int ii = seg_lo + (warp - seg_lo % kConsumerWarps + kConsumerWarps) % kConsumerWarps; ii < seg_hi;
         ii += kPair * kConsumerWarps) {
      const bool two = kPair == 2 && ii + kConsumerWarps < seg_hi;
      const int k = ii / kConsumerWarps;
      advance(k);
      const int nt0 = nt_of(k);
      int nt1 = 0;
      if (two) {
        advance(k + 1);
        nt1 = nt_of(k + 1);
      }
      const int st0 = ii % C::kStages, st1 = (ii + kConsumerWarps) % C::kStages;
      const uint32_t ph0 = (uint32_t)(k / C::kPerWarp) & 1u, ph1 = (uint32_t)((k + 1) / C::kPerWarp) & 1u;
      int nrow, nnt;  // the page (of the next ones) whose halves this lane refills
      where(k, two ? 2 : 1, nrow, nnt);
      bool got = ok && mbar_wait(&kfull[st0], ph0);
      if (got && two) got = mbar_wait(&kfull[st1], ph1);
      if (ok && !got) {
        if (lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
        ok = false;  // a copy may still be in flight: issue nothing more
      }
      const uint32_t kb0 = ring_s + st0 * C::kStageBytes, kb1 = ring_s + st1 * C::kStageBytes;
      constexpr int MT = C::PS / 16;
      float sc[2 * MT][4];  // the scores of one or two pages
      const bool pair = two && nt0 > 0 && nt1 > 0;  // both pages in one pass
      if (got) {
        if (pair) {
          const uint32_t kbs[2] = {kb0, kb1};
          const int nts[2] = {nt0, nt1};
          attend_scores<C::PS, 2>(kbs, nts, qa, a.scale_log2, sc, lane);
        } else {
          const int ntx = nt0 > 0 ? nt0 : nt1;  // the one page with tokens (if any)
          const uint32_t kbs[1] = {nt0 > 0 ? kb0 : kb1};
          const int nts[1] = {ntx};
          if (ntx > 0) attend_scores<C::PS, 1>(kbs, nts, qa, a.scale_log2, reinterpret_cast<float(&)[MT][4]>(sc), lane);
        }
      }
      // the K halves may be reloaded once every lane has read them (ldmatrix only: those reads
      // returned before the MMAs that use them issued, so no proxy fence is needed)
      if (ok) {
        __syncwarp();
        refill(k, two ? 2 : 1, nrow, nnt, 0);
      }
      if (got) {
        got = mbar_wait(&vfull[st0], ph0);
        if (got && two) got = mbar_wait(&vfull[st1], ph1);
        if (ok && !got) {
          if (lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
          ok = false;
        }
      }
      bool cleared = false;  // generic stores went into a V half (warp-uniform)
      if (got) {
        if (nt0 > 0 && nt0 < C::PS) {
          clear_tail_rows<C::PS>(ring + st0 * C::kStageBytes + 2 * C::kHalfBytes, nt0, lane);
          cleared = true;
        }
        if (two && nt1 > 0 && nt1 < C::PS) {
          clear_tail_rows<C::PS>(ring + st1 * C::kStageBytes + 2 * C::kHalfBytes, nt1, lane);
          cleared = true;
        }
        if (pair) {
          const uint32_t vbs[2] = {kb0 + 2 * C::kHalfBytes, kb1 + 2 * C::kHalfBytes};
          attend_values<C::PS, 2>(vbs, sc, st, lane);
        } else if (nt0 > 0 || (two && nt1 > 0)) {
          const uint32_t vbs[1] = {(nt0 > 0 ? kb0 : kb1) + 2 * C::kHalfBytes};
          attend_values<C::PS, 1>(vbs, reinterpret_cast<float(&)[MT][4]>(sc), st, lane);
        }
      }
      // and the V halves once P V is done; zeroed tail rows are generic writes, which the copy
      // that overwrites them must be ordered after
      if (ok) {
        if (cleared) fence_proxy_async();
        __syncwarp();
        refill(k, two ? 2 : 1, nrow, nnt, 1);
      }
    }
    i = seg_hi;
    // hand this warp's state for the segment to the epilogue warp
    float l0 = st.l[0], l1 = st.l[1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const int slot = sg % a.nslots;
    if (!mbar_wait(&cempty[slot], ((uint32_t)(sg / a.nslots) & 1u) ^ 1u) && lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
    const SlotView<NC> cs{cbf + slot * slot_f, a.G};
    if (g == 0) {
      if (2 * t < a.G) {
        cs.m(warp, 2 * t) = st.m[0];
        cs.l(warp, 2 * t) = l0;
      }
      if (2 * t + 1 < a.G) {
        cs.m(warp, 2 * t + 1) = st.m[1];
        cs.l(warp, 2 * t + 1) = l1;
      }
    }
#pragma unroll
    for (int md = 0; md < 8; ++md) {
      const int d0 = md * 16 + g;
      if (2 * t < a.G) {
        cs.o(warp, 2 * t)[d0] = st.o[md][0];
        cs.o(warp, 2 * t)[d0 + 8] = st.o[md][2];
      }
      if (2 * t + 1 < a.G) {
        cs.o(warp, 2 * t + 1)[d0] = st.o[md][1];
        cs.o(warp, 2 * t + 1)[d0 + 8] = st.o[md][3];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&cfull[slot]);
    have = it.next(u, lo, hi);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = qn[ks][0];
      qa[ks][1] = qn[ks][1];
    }
  }
  // this CTA's pages are done: a kernel that starts early after this one may take the SMs the
  // grid leaves while the epilogue and split warps finish
  release_dependents();
}

inline size_t counters_bytes(int64_t units) { return (size_t)((units * 4 + 255) / 256 * 256); }
constexpr size_t kSlotLseBytes = (size_t)kMaxGrid * 2 * kMaxG * sizeof(float);
constexpr size_t kSlotOBytes = (size_t)kMaxGrid * 2 * kMaxG * kD * sizeof(float);

template <int P, int S, int NC>
size_t dyn_smem(int units, int G, int nslots) {
  return 1024 + Cfg<P, S, NC>::kRingBytes + (size_t)nslots * slot_floats(G, NC) * sizeof(float) +
         (size_t)(units + 1) * 4;
}
constexpr size_t kSmemLimit = 232448 - 1024;  // per-block shared memory minus room for static use




// The pool [n_slots * P rows][128 columns] bf16 seen as a 3-D tensor [2 halves][rows][64
// columns] (half stride 128 bytes, row stride 256 bytes): one box {64, box_rows, 2} is a whole
// sub-page, landing in shared memory as two [box_rows][64] halves with the 128-byte swizzle.
bool make_page_map(CUtensorMap* map, const void* pool, int64_t n_slots, int P, int box_rows) {
  const cuuint64_t dims[3] = {64, (cuuint64_t)(n_slots * P), 2};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
                      CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS;
}

template <int P, int S, int NC, bool UNITS>
bool prepare(size_t smem) {
  auto kern = sparse_attn_kernel<P, S, NC, UNITS>;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess &&
         cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess;
}

template <int P, int S, int NC, bool UNITS>
int launch_grid(const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnArgs& a, const scout_launch* launch,
                int grid, size_t smem, cudaStream_t stream) {
  constexpr int kThreads = threads_of<NC>();
  auto kern = sparse_attn_kernel<P, S, NC, UNITS>;
  if (UNITS && !prepare<P, S, NC, UNITS>(smem)) return SCOUT_ERR_CUDA;  // the other one was prepared for the query
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = early_start_attrs(launch, attr, 0);
  if (cudaLaunchKernelEx(&cfg, kern, tmK, tmV, a) != cudaSuccess) return SCOUT_ERR_CUDA;
  return launch_status();
}

// One CTA per SM (or the caller's cap); the instance that may take whole units when the grid
// covers them.
template <int P, int S, int NC>
int launch_ring(const CUtensorMap& tmK, const CUtensorMap& tmV, AttnArgs a, const scout_launch* launch,
                cudaStream_t stream) {
  const int max_ctas = launch != nullptr ? launch->max_ctas : 0;
  const size_t smem = dyn_smem<P, S, NC>(a.units, a.G, a.nslots);
  int occ = 0;
  if (!prepare<P, S, NC, false>(smem) ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparse_attn_kernel<P, S, NC, false>, threads_of<NC>(),
                                                    smem) != cudaSuccess ||
      occ < 1)
    return SCOUT_ERR_CUDA;
  const int grid = min(kMaxGrid, max_ctas > 0 ? max_ctas : sm_count() * occ);
  return a.units <= grid ? launch_grid<P, S, NC, true>(tmK, tmV, a, launch, grid, smem, stream)
                         : launch_grid<P, S, NC, false>(tmK, tmV, a, launch, grid, smem, stream);
}

// The most combine slots that fit with ring S and NC consumer warps; 0 if none does.
template <int P, int S, int NC>
int slots_fitting(const AttnArgs& a) {
  for (int ns = kMaxSlots; ns >= 1; --ns)
    if (dyn_smem<P, S, NC>(a.units, a.G, ns) <= kSmemLimit) return ns;
  return 0;
}

// The first configuration that fits in shared memory, with the most combine slots it allows:
// the preferred consumer warps with the whole ring, then four warps with the whole ring (their
// combine state is smaller), then four warps with the smaller ring.
template <int P>
int launch_attn(const void* K_pool, const void* V_pool, AttnArgs a, const scout_launch* launch, cudaStream_t stream) {
  constexpr int NA = kConsumers, NB = kFallbackConsumers;
  constexpr int SA = big_ring<P, NA>(), SB = big_ring<P, NB>(), SC = small_ring<P, NB>();
  constexpr int PS = Cfg<P, SA, NA>::PS;
  static_assert(Cfg<P, SB, NB>::PS == PS && Cfg<P, SC, NB>::PS == PS, "one stage size for all rings");
  CUtensorMap tmK, tmV;
  if (!make_page_map(&tmK, K_pool, a.n_slots, P, PS) || !make_page_map(&tmV, V_pool, a.n_slots, P, PS))
    return SCOUT_ERR_UNSUPPORTED;
  if ((a.nslots = slots_fitting<P, SA, NA>(a)) > 0) return launch_ring<P, SA, NA>(tmK, tmV, a, launch, stream);
  if ((a.nslots = slots_fitting<P, SB, NB>(a)) > 0) return launch_ring<P, SB, NB>(tmK, tmV, a, launch, stream);
  if ((a.nslots = slots_fitting<P, SC, NB>(a)) > 0) return launch_ring<P, SC, NB>(tmK, tmV, a, launch, stream);
  return SCOUT_ERR_UNSUPPORTED;
}

// Shared by both entry points: O_part/lse_part for the partial, or (O_cpu, lse_cpu,
// O_out, lse_out) for the merged output.
int attn_entry(const void* q, const void* K_pool, const void* V_pool, int64_t n_slots, const int32_t* page_table,
               const int32_t* seq_len, const int32_t* res_list, const int32_t* res_count, int B, int Hq, int Hkv,
               int D, int P, int nblk_cap, int k, float scale, float* O_part, float* lse_part, const float* O_cpu,
               const float* lse_cpu, __nv_bfloat16* O_out, float* lse_out, void* workspace,
               size_t workspace_bytes, int32_t* dev_status, const scout_launch* launch, cudaStream_t stream) {
  const bool merge = O_out != nullptr;
  if (q == nullptr || K_pool == nullptr || V_pool == nullptr || page_table == nullptr || seq_len == nullptr ||
      res_list == nullptr || res_count == nullptr)
    return SCOUT_ERR_INVALID_ARG;
  if (merge ? (O_cpu == nullptr || lse_cpu == nullptr) : (O_part == nullptr || lse_part == nullptr))
    return SCOUT_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || n_slots <= 0 || nblk_cap <= 0 || k <= 0 ||
      !(scale > 0.f))
    return SCOUT_ERR_INVALID_ARG;
  if (launch != nullptr && launch->max_ctas < 0) return SCOUT_ERR_INVALID_ARG;
  const int64_t units = (int64_t)B * Hkv;
  const int G = Hq / Hkv;
  if (D != kD || !valid_P(P) || G > kMaxG || units > kMaxUnits || !aligned16(K_pool) || !aligned16(V_pool) ||
      (reinterpret_cast<uintptr_t>(q) & 3u) || n_slots * P > (int64_t)0x7fffffff || units * k > kMaxEntries)
    return SCOUT_ERR_UNSUPPORTED;
  if (merge && (!aligned16(O_cpu) || (reinterpret_cast<uintptr_t>(O_out) & 7u))) return SCOUT_ERR_UNSUPPORTED;
  if (!merge && !aligned16(O_part)) return SCOUT_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < scout_sparse_attn_workspace_bytes(B, Hq, Hkv, D, P))
    return SCOUT_ERR_WORKSPACE;
  AttnArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.page_table = page_table;
  a.seq_len = seq_len;
  a.res_list = res_list;
  a.res_count = res_count;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.nblk_cap = nblk_cap;
  a.k = k;
  a.units = (int)units;
  a.n_slots = n_slots;
  a.scale_log2 = scale * kLog2e;
  a.O_part = O_part;
  a.lse_part = lse_part;
  a.O_cpu = O_cpu;
  a.lse_cpu = lse_cpu;
  a.O_out = O_out;
  a.lse_out = lse_out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.counters = reinterpret_cast<int32_t*>(ws);
  a.slot_lse = reinterpret_cast<float*>(ws + counters_bytes(units));
  a.slot_O = reinterpret_cast<float*>(ws + counters_bytes(units) + kSlotLseBytes);
  a.status = dev_status;
  switch (P) {
    case 16: return launch_attn<16>(K_pool, V_pool, a, launch, stream);
    case 32: return launch_attn<32>(K_pool, V_pool, a, launch, stream);
    default: return launch_attn<64>(K_pool, V_pool, a, launch, stream);
  }
}

}  // namespace
}  // namespace scout

extern "C" size_t scout_sparse_attn_workspace_bytes(int B, int Hq, int Hkv, int D, int P) {
  (void)Hq;
  (void)D;
  (void)P;
  if (B <= 0 || Hkv <= 0) return 0;
  return scout::counters_bytes((int64_t)B * Hkv) + scout::kSlotLseBytes + scout::kSlotOBytes;
}

extern "C" int scout_sparse_attn(const void* q, const void* K_pool, const void* V_pool, int64_t n_slots,
                                 const int32_t* page_table, const int32_t* seq_len, const int32_t* res_list,
                                 const int32_t* res_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap, int k,
                                 float scale, float* O_part, float* lse_part, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, const scout_launch* launch, cudaStream_t stream) {
  if (O_part == nullptr || lse_part == nullptr) return SCOUT_ERR_INVALID_ARG;
  return scout::attn_entry(q, K_pool, V_pool, n_slots, page_table, seq_len, res_list, res_count, B, Hq, Hkv, D, P,
                           nblk_cap, k, scale, O_part, lse_part, nullptr, nullptr, nullptr, nullptr, workspace,
                           workspace_bytes, dev_status, launch, stream);
}

extern "C" int scout_sparse_attn_merge(const void* q, const void* K_pool, const void* V_pool, int64_t n_slots,
                                       const int32_t* page_table, const int32_t* seq_len, const int32_t* res_list,
                                       const int32_t* res_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap,
                                       int k, float scale, const float* O_cpu, const float* lse_cpu, void* O_out,
                                       float* lse_out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                       const scout_launch* launch, cudaStream_t stream) {
  if (O_out == nullptr) return SCOUT_ERR_INVALID_ARG;
  return scout::attn_entry(q, K_pool, V_pool, n_slots, page_table, seq_len, res_list, res_count, B, Hq, Hkv, D, P,
                           nblk_cap, k, scale, nullptr, nullptr, O_cpu, lse_cpu,
                           static_cast<__nv_bfloat16*>(O_out), lse_out, workspace, workspace_bytes, dev_status,
                           launch, stream);
}
