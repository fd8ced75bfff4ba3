// scout_score_topk: digest scoring, per-unit top-k, residency split, CPU work list.
// ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1: B_pred = TopK(q K_digest^T),
// B_cpu = B_pred \ B_gpu.
//
// One persistent, warp-specialised kernel (one CTA per SM):
//  * warp 12 streams work items (unit, 128-row digest chunk) with TMA: four 128-byte
//    swizzled boxes of the chunk plus the unit's query rows, into a ring of stages;
//  * warps 0..7 score one 16-row tile of each chunk on the tensor cores.  A score is a
//    dot product over the 256 [min | max] digest values (q- pairs with min, q+ with
//    max) or over the 128 fp32 means split exactly into three bf16 terms, so mma.sync
//    with bf16 operands and fp32 accumulation computes it (products are exact).  The
//    score pooled over the unit's G query heads (maximum) becomes an orderable key in
//    shared memory;
//  * warps 8..11 select the units as their chunks are scored, one warp per unit and up
//    to four units at a time: radix select of the k-th key, then one ordered compaction
//    into top-k, resident, CPU and delta lists.
// Whole units are dealt out to the CTAs one at a time from a ticket counter in the
// workspace: a unit is always scored and selected inside one CTA, and a CTA that starts
// late (its SM was still busy with another kernel when the grid launched) or draws short
// units takes more of them, so a grid of one CTA per SM fills SMs as they free up.
#include <mutex>

#include "common.cuh"

namespace scout {
namespace {

constexpr int kScoreWarps = 8;
constexpr int kSelWarps = 4;
constexpr int kProducer = kScoreWarps + kSelWarps;  // warp index of the TMA producer
constexpr int kThreadsAll = (kProducer + 1) * 32;
constexpr int kChunk = kScoreWarps * 16;  // digest rows (blocks) per work item
constexpr int kBoxBytes = kChunk * 128;   // one 128-row x 128-byte TMA box
constexpr int kMaxStagesT = 3;
constexpr int kMaxKeyBufs = 8;  // key buffers: one being scored, the others being selected
constexpr int kSeqCache = 256;  // sequence lengths kept in shared memory (larger batches read the rest)

__device__ __forceinline__ uint32_t trunc_bf16(float x) { return __float_as_uint(x) & 0xFFFF0000u; }

// Orderable key of an fp32 score: larger score -> larger key; -0 and +0 equal.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t b = __float_as_uint(s == 0.f ? 0.f : s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The query group sits in shared memory with rows kQStride bf16 apart (272 bytes):
// the 8 rows a fragment load touches then fall on distinct banks.
constexpr int kQStride = kD + 8;
constexpr int kQBytes = kMaxG * kQStride * 2;
// digest chunk + the unit's query group, rounded so every stage starts 1024-aligned
constexpr int kStageBytesT = (4 * kBoxBytes + kQBytes + 1023) / 1024 * 1024;

// Keep the bf16 halves of a pair whose sign bit is clear (q+) or set (q-).
__device__ __forceinline__ uint32_t pos_part(uint32_t v) { return v & ~(((v >> 15) & 0x00010001u) * 0xFFFFu); }
__device__ __forceinline__ uint32_t neg_part(uint32_t v) { return v & (((v >> 15) & 0x00010001u) * 0xFFFFu); }

// q fragment (B operand) for the min/max kind, standard k order: k-step s covers
// digest values [16 s, 16 s + 16) of the [min | max] row, i.e. part s / 8 (min pairs
// with q-, max with q+) and channels (s % 8) * 16 + {2t, 2t+1, 2t+8, 2t+9}.
__device__ __forceinline__ void minmax_b_frag(const __nv_bfloat16* qs, int G, int lane, uint32_t (&bf)[16][2]) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t* row = reinterpret_cast<const uint32_t*>(qs + g * kQStride);
#pragma unroll
  for (int s8 = 0; s8 < 8; ++s8) {
    const uint32_t lo = g < G ? row[s8 * 8 + t] : 0u, hi = g < G ? row[s8 * 8 + t + 4] : 0u;
    bf[s8][0] = neg_part(lo);
    bf[s8][1] = neg_part(hi);
    bf[s8 + 8][0] = pos_part(lo);
    bf[s8 + 8][1] = pos_part(hi);
  }
}

// q fragment for the mean kind: load i of lane t covers channels i*16 + t*4 + {0..3}.
__device__ __forceinline__ void mean_b_frag(const __nv_bfloat16* qs, int G, int lane, uint32_t (&bf)[8][2]) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t* row = reinterpret_cast<const uint32_t*>(qs + g * kQStride);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    bf[i][0] = g < G ? row[i * 8 + 2 * t] : 0u;
    bf[i][1] = g < G ? row[i * 8 + 2 * t + 1] : 0u;
  }
}

// A chunk of 128 digest rows sits in shared memory as four TMA boxes of
// 128 rows x 128 bytes (row bytes [128 b, 128 b + 128) in box b), each with the
// 128-byte swizzle: 16-byte chunk c of row r lives at chunk c ^ (r % 8).
//   address(r, C) = (C >> 3) * kBoxBytes + r * 128 + (((C & 7) ^ (r & 7)) << 4).
// A scoring warp reads rows r0 + (lane part) whose r & 7 is a lane constant, at chunks
// C = c + (a lane part smaller than the step of c) + 8 box, so each address is a per-lane offset
// (one of four for the min/max digest, two for the mean) plus box * kBoxBytes, computed once.
struct TileOfs {
  uint32_t o[4];
};
// min/max: ldmatrix rows r0 + 8 ((lane >> 3) & 1) + (lane & 7), chunks 2 s + (lane >> 4):
// o[i] covers c = 2 i (s & 3 = i), box s >> 2
__device__ __forceinline__ TileOfs minmax_offsets(int r0, int lane) {
  TileOfs t;
  const uint32_t l7 = lane & 7, r = r0 + ((lane >> 3) & 1) * 8 + l7, hb = lane >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) t.o[i] = r * 128 + (((2u * i) ^ hb ^ l7) << 4);
  return t;
}
// mean: rows r0 + g (and r0 + g + 8, 1024 bytes further), chunks 4 i + t: o[i & 1] covers
// c = 4 (i & 1), box i >> 1
__device__ __forceinline__ TileOfs mean_offsets(int r0, int lane) {
  TileOfs t;
  const uint32_t g = lane >> 2, tt = lane & 3;
#pragma unroll
  for (int i = 0; i < 2; ++i) t.o[i] = (r0 + g) * 128 + (((4u * i) ^ tt ^ g) << 4);
  t.o[2] = t.o[3] = 0u;
  return t;
}

// Scores of the warp's 16 rows (local rows r0 .. r0 + 15): c = rows g, g + 8 x heads 2t, 2t+1.
template <int KIND>
__device__ __forceinline__ void score_tile(uint32_t tbase, const TileOfs& to, const uint32_t (&bmm)[16][2],
                                           const uint32_t (&bme)[8][2], float (&c)[4]) {
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  if (KIND == SCOUT_DIGEST_MINMAX) {
#pragma unroll
    for (int s = 0; s < 16; ++s) {  // four independent accumulation chains
      uint32_t a0, a1, a2, a3;
      ldsm_x4(tbase + to.o[s & 3] + (s >> 2) * kBoxBytes, a0, a1, a2, a3);
      mma_bf16(acc[s & 3], a0, a1, a2, a3, bmm[s][0], bmm[s][1]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // four fp32 channels i*16 + 4t .. +3 of rows g and g + 8, split exactly as hi + mid + lo (bf16)
      uint4 v0, v1;
      const uint32_t p0 = tbase + to.o[i & 1] + (i >> 1) * kBoxBytes, p1 = p0 + 8 * 128;
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v0.x), "=r"(v0.y), "=r"(v0.z), "=r"(v0.w) : "r"(p0));
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v1.x), "=r"(v1.y), "=r"(v1.z), "=r"(v1.w) : "r"(p1));
      const float x0[4] = {__uint_as_float(v0.x), __uint_as_float(v0.y), __uint_as_float(v0.z), __uint_as_float(v0.w)};
      const float x1[4] = {__uint_as_float(v1.x), __uint_as_float(v1.y), __uint_as_float(v1.z), __uint_as_float(v1.w)};
      float r0v[4], r1v[4];
      uint32_t h0[4], h1[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h0[e] = trunc_bf16(x0[e]);
        h1[e] = trunc_bf16(x1[e]);
        r0v[e] = x0[e] - __uint_as_float(h0[e]);
        r1v[e] = x1[e] - __uint_as_float(h1[e]);
      }
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        uint32_t a0[4], a1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (part == 0) {
            a0[e] = h0[e];
            a1[e] = h1[e];
          } else if (part == 1) {
            a0[e] = trunc_bf16(r0v[e]);
            a1[e] = trunc_bf16(r1v[e]);
          } else {
            a0[e] = trunc_bf16(r0v[e] - __uint_as_float(trunc_bf16(r0v[e])));
            a1[e] = trunc_bf16(r1v[e] - __uint_as_float(trunc_bf16(r1v[e])));
          }
        }
        // pack two bf16 (upper halves of the fp32 patterns): low half = lower k
        const uint32_t A0 = (a0[0] >> 16) | a0[1], A1 = (a1[0] >> 16) | a1[1];
        const uint32_t A2 = (a0[2] >> 16) | a0[3], A3 = (a1[2] >> 16) | a1[3];
        mma_bf16(acc[part], A0, A1, A2, A3, bme[i][0], bme[i][1]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) c[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
}

struct TopkArgs {
  const __nv_bfloat16* q;
  const uint8_t* digest;
  const int32_t* seq_len;
  const uint32_t* resident_bits;
  const int32_t* prev_list;
  const int32_t* prev_count;
  int Hq, Hkv, G, P, nblk_cap, k, words, nchunk, stages;
  int nkbuf;  // key buffers in shared memory (2 .. kMaxKeyBufs)
  int nsel;   // selector warps in use (1 .. min(kSelWarps, nkbuf - 1))
  int user_scores;  // 1: the caller asked for every pooled score in `scores`
  int units;
  float* scores;  // the caller's buffer, written only when user_scores
  int32_t* counters;  // [0]: the unit ticket counter (zero between calls)
  int32_t* status;
  uint32_t score_wait;  // poll limit of the scoring warps' waits for a stage to land
  int inject;           // SCOUT_INJECT_* (tests)
  int32_t *topk_idx, *topk_count, *res_list, *res_count, *cpu_list, *cpu_count, *delta_list, *delta_count;
};

__host__ __device__ constexpr int align4(int n) { return (n + 3) / 4 * 4; }  // words to a 16-byte multiple


// A selector warp's shared memory: the unit's residency bits, the bits of its previous
// CPU list, the bits of the chosen candidates, a 256-bin digit histogram and the blocks
// of up to kMaxCand candidates.
struct SelWarp {
  uint32_t* rbits;  // [words]
  uint32_t* pbits;  // [words]
  uint32_t* cbits;  // [words]
  int* hist;        // [256]
  int* cidx;        // [kMaxCand]
};
// 32-bit words of one selector warp's shared memory
constexpr int kMaxCand = 64;  // candidates ranked exactly in the warp (two per lane)
__host__ __device__ constexpr int selwarp_words(int words) { return 3 * align4(words) + 256 + kMaxCand; }
__device__ __forceinline__ SelWarp selwarp_at(uint32_t* area, int words) {
  const int w4 = align4(words);
  return SelWarp{area, area + w4, area + 2 * w4, reinterpret_cast<int*>(area + 3 * w4),
                 reinterpret_cast<int*>(area + 3 * w4 + 256)};
}

// Loads the unit's residency bits and previous CPU list into the warp's shared memory.
__device__ void prefetch_unit(const TopkArgs& a, int u, const SelWarp& sw, int lane) {
  for (int i = lane; i < a.words; i += 32) {
    sw.rbits[i] = a.resident_bits[(int64_t)u * a.words + i];
    sw.pbits[i] = 0u;
  }
  __syncwarp();
  if (a.prev_list != nullptr) {
    const int pc = min(max(a.prev_count[u], 0), a.k);
    for (int i = lane; i < pc; i += 32) {
      const int j = a.prev_list[(int64_t)u * a.k + i];
      if (j >= 0 && j < a.nblk_cap) atomicOr(&sw.pbits[j >> 5], 1u << (j & 31));
    }
  }
  __syncwarp();
}

// Keys g0 + 32 r + lane (r = 0..31) of a group of 1024, minus base, into registers
// (0 past nvalid).
__device__ __forceinline__ void load_group(const uint32_t* keys, int nvalid, int g0, int lane, uint32_t (&kv)[32],
                                           uint32_t base = 0u) {
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const int j = g0 + 32 * r + lane;
    kv[r] = j < nvalid ? keys[j] - base : 0u;
  }
}

// 32 x 32 bit transpose across a warp: bit j of lane i's word becomes bit i of lane j's
// word (block swaps of 16, 8, 4, 2 and 1).
__device__ __forceinline__ uint32_t transpose32(uint32_t x, int lane) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    const uint32_t m = s == 16 ? 0x0000FFFFu : s == 8 ? 0x00FF00FFu : s == 4 ? 0x0F0F0F0Fu : s == 2 ? 0x33333333u
                                                                                                     : 0x55555555u;
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, s);
    x = (lane & s) ? ((x & ~m) | ((y & ~m) >> s)) : ((x & m) | ((y & m) << s));
  }
  return x;
}

// Exclusive prefix sums over the lanes of two counts (each < 2^15 in total) with one scan:
// the counts travel as the two 16-bit halves of one word.  Also returns the totals.
__device__ __forceinline__ void scan_pair(int x, int y, int lane, int& ex, int& ey, int& tx, int& ty) {
  const int v = x | (y << 16);
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int z = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += z;
  }
  const int tot = __shfl_sync(0xffffffffu, incl, 31), e = incl - v;
  ex = e & 0xffff;
  ey = e >> 16;
  tx = tot & 0xffff;
  ty = tot >> 16;
}

// Top-k of one unit's keys (shared memory), split by residency, delta against the previous
// CPU list, written in ascending block order.  One warp, no block-level barrier.
//
// The keys are taken 1024 at a time into registers (lane l holds keys 32 r + l), so every
// step is a run of independent instructions.  The k-th largest key is bracketed by a radix
// select on key - min: the leading bits zero in all of them are skipped, then 8-bit digits
// of the keys sharing the current prefix are counted into a 256-bin histogram (shared-memory
// reductions) until the keys sharing the prefix (the candidates) are the ones still needed
// or at most 64.  Keys above the prefix are selected.  Of the candidates the `remaining`
// largest are taken, the lower block index first among equal keys: with at most 64 of them
// each lane ranks two against all the others; more can only be left when every candidate
// key is equal, and then the lowest-index ones are taken.  The chosen candidates go into a
// bitmap.  Per-round bit masks move between "lane = block" and "lane = round" by a 32 x 32
// bit transpose, so no step needs a shuffle per round; lane r then writes round r's blocks
// at the list positions two packed prefix scans give it.
__device__ void select_unit(const TopkArgs& a, int u, const uint32_t* keys, int nvalid, const SelWarp& sw,
                            int lane) {
  const int keff = min(a.k, nvalid);
  const int ngroups = (nvalid + 1023) / 1024;
  uint32_t kv[32];
  if (ngroups == 1) load_group(keys, nvalid, 0, lane, kv);  // stays in registers throughout
  uint32_t prefix = 0u, mask = 0u, base = 0u;  // selection works on key - base
  int remaining = keff, count = nvalid;
  if (keff < nvalid) {
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int g = 0; g < ngroups; ++g) {
      if (ngroups > 1) load_group(keys, nvalid, g * 1024, lane, kv);
#pragma unroll
      for (int r = 0; r < 32; ++r)
        if (g * 1024 + 32 * r + lane < nvalid) {
          lo = min(lo, kv[r]);
          hi = max(hi, kv[r]);
        }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    // relative keys keep the order; their digits start at the top bit of the key range, so
    // the first digit already spreads the keys over the bins
    base = lo;
    if (ngroups == 1) {
#pragma unroll
      for (int r = 0; r < 32; ++r) kv[r] -= base;
    }
    int fixed = lo == hi ? 32 : __clz(hi - lo);  // leading bits zero in every relative key
    mask = fixed == 0 ? 0u : (fixed == 32 ? 0xffffffffu : ~(0xffffffffu >> fixed));
    int4* h4 = reinterpret_cast<int4*>(sw.hist);
    while (fixed < 32 && remaining != count && count > kMaxCand) {
      const int width = min(8, 32 - fixed), shift = 32 - fixed - width;
      const uint32_t dmask = (1u << width) - 1u;
      h4[lane] = make_int4(0, 0, 0, 0);
      h4[lane + 32] = make_int4(0, 0, 0, 0);
      __syncwarp();
      for (int g = 0; g < ngroups; ++g) {
        if (ngroups > 1) load_group(keys, nvalid, g * 1024, lane, kv, base);
#pragma unroll
        for (int r = 0; r < 32; ++r)
          if (g * 1024 + 32 * r + lane < nvalid && (kv[r] & mask) == prefix)
            atomicAdd(&sw.hist[(kv[r] >> shift) & dmask], 1);
      }
      __syncwarp();
      // lane L holds bins 8L .. 8L+7; counts above each lane from the highest bin down
      const int4 x0 = h4[2 * lane], x1 = h4[2 * lane + 1];
      const int c8[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const int own = x0.x + x0.y + x0.z + x0.w + x1.x + x1.y + x1.z + x1.w;
      int suf = own;  // bins >= 8L
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += y;
      }
      const int above = suf - own;  // bins > 8L + 7
      const int L = __ffs(__ballot_sync(0xffffffffu, above < remaining && remaining <= suf)) - 1;
      int digit = 0, rem = 0, cnt = 0;
      if (lane == L) {
        int acc = above;
#pragma unroll
        for (int e = 7; e >= 0; --e) {
          if (acc < remaining && remaining <= acc + c8[e] && cnt == 0) {
            digit = 8 * L + e;
            rem = remaining - acc;
            cnt = c8[e];
          }
          acc += c8[e];
        }
      }
      __syncwarp();  // every lane has read the histogram before it is reused
      prefix |= (uint32_t)__shfl_sync(0xffffffffu, digit, L) << shift;
      mask |= dmask << shift;
      remaining = __shfl_sync(0xffffffffu, rem, L);
      count = __shfl_sync(0xffffffffu, cnt, L);
      fixed += width;
    }
  }
  const bool all_eq = remaining == count;  // every candidate is taken
  if (!all_eq) {
    for (int i = lane; i < a.words; i += 32) sw.cbits[i] = 0u;
    __syncwarp();
    const uint32_t lt = (1u << lane) - 1u;
    if (count <= kMaxCand) {
      // gather the candidates in block order (lane r takes round r of each group of 1024 after a
      // bit transpose), then one per lane ranks itself against the others
      int n = 0;
      for (int g = 0; g < ngroups; ++g) {
        if (ngroups > 1) load_group(keys, nvalid, g * 1024, lane, kv, base);
        uint32_t e = 0u;  // bit r: this lane's key of round r is a candidate
#pragma unroll
        for (int r = 0; r < 32; ++r)
          if (g * 1024 + 32 * r + lane < nvalid && (kv[r] & mask) == prefix) e |= 1u << r;
        uint32_t em = transpose32(e, lane);  // candidates of round `lane`
        const int c = __popc(em);
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        for (int pos = n + incl - c; em != 0u; ++pos, em &= em - 1u) sw.cidx[pos] = g * 1024 + 32 * lane + __ffs(em) - 1;
        n += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncwarp();
      // lane l ranks candidates l and l + 32 against all of them
      const int j0 = lane < count ? sw.cidx[lane] : 0, j1 = lane + 32 < count ? sw.cidx[lane + 32] : 0;
      const uint32_t k0 = lane < count ? keys[j0] - base : 0u, k1 = lane + 32 < count ? keys[j1] - base : 0u;
      int r0 = 0, r1 = 0;
      for (int h = 0; h < (count + 31) / 32; ++h) {
        const int mmax = min(32, count - 32 * h);  // warp-uniform: only the candidates there are
        for (int m = 0; m < mmax; ++m) {
          const uint32_t km = __shfl_sync(0xffffffffu, h ? k1 : k0, m);
          const int jm = __shfl_sync(0xffffffffu, h ? j1 : j0, m);
          r0 += (km > k0 || (km == k0 && jm < j0)) ? 1 : 0;
          r1 += (km > k1 || (km == k1 && jm < j1)) ? 1 : 0;
        }
      }
      if (lane < count && r0 < remaining) atomicOr(&sw.cbits[j0 >> 5], 1u << (j0 & 31));
      if (lane + 32 < count && r1 < remaining) atomicOr(&sw.cbits[j1 >> 5], 1u << (j1 & 31));
    } else {
      // more than kMaxCand candidates are left only when all of them are equal: the lowest-index ones
      int seen = 0;
      for (int g = 0; g < ngroups; ++g) {
        if (ngroups > 1) load_group(keys, nvalid, g * 1024, lane, kv, base);
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          const int j = g * 1024 + 32 * r + lane;
          const bool eq = j < nvalid && (kv[r] & mask) == prefix;
          const uint32_t eqb = __ballot_sync(0xffffffffu, eq);
          const uint32_t sb = __ballot_sync(0xffffffffu, eq && seen + __popc(eqb & lt) < remaining);
          if (lane == 0) sw.cbits[g * 32 + r] = sb;
          seen += __popc(eqb);
        }
      }
    }
    __syncwarp();
  }
  // compaction: per lane one bit per round, transposed so that lane r holds round r's
  // selected blocks; each list is then written with coalesced stores
  const int64_t lb = (int64_t)u * a.k;
  int nt = 0, nr = 0, nc = 0, nd = 0;
  for (int g = 0; g < ngroups; ++g) {
    if (ngroups > 1) load_group(keys, nvalid, g * 1024, lane, kv, base);
    const int w = g * 32 + lane;  // word of round `lane` in the per-block bitmaps
    const uint32_t rw = w < a.words ? sw.rbits[w] : 0u, pw = w < a.words ? sw.pbits[w] : 0u;
    // bit r of tb: the candidate at (round r, this lane) is taken
    const uint32_t tb = all_eq ? 0xffffffffu : transpose32(w < a.words ? sw.cbits[w] : 0u, lane);
    uint32_t sel = 0u;  // bit r: this lane's block of round r is selected
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const uint32_t mk = kv[r] & mask;
      if (g * 1024 + 32 * r + lane < nvalid && (mk > prefix || (mk == prefix && ((tb >> r) & 1u)))) sel |= 1u << r;
    }
    const uint32_t ms = transpose32(sel, lane);  // selected blocks of round `lane`
    const uint32_t mres = ms & rw, mcpu = ms & ~rw, mdel = ms & ~rw & ~pw;
    // lane r writes its round's blocks; two packed scans give every lane's list positions
    int et, er, ec, ed, tt, tr, tc, td;
    scan_pair(__popc(ms), __popc(mres), lane, et, er, tt, tr);
    scan_pair(__popc(mcpu), __popc(mdel), lane, ec, ed, tc, td);
    const int j0 = g * 1024 + 32 * lane;
    // one pass over the round's selected blocks in order: every block goes to top-k and to the
    // resident or the CPU list, and a CPU block that was not on the previous list to delta
    int32_t* const tl = a.topk_idx + lb;
    int32_t* const rl = a.res_list + lb;
    int32_t* const cl = a.cpu_list + lb;
    int32_t* const dl = a.delta_list + lb;
    int qt = nt + et, qr = nr + er, qc = nc + ec, qd = nd + ed;
    for (uint32_t m = ms; m != 0u; m &= m - 1u) {
      const int bit = __ffs(m) - 1;
      const uint32_t one = 1u << bit;
      const int j = j0 + bit;
      tl[qt++] = j;
      if (rw & one) {
        rl[qr++] = j;
      } else {
        cl[qc++] = j;
        if (!(pw & one)) dl[qd++] = j;
      }
    }
    nt += tt;
    nr += tr;
    nc += tc;
    nd += td;
  }
  for (int i = lane; i < a.k; i += 32) {
    if (i >= nt) a.topk_idx[lb + i] = -1;
    if (i >= nr) a.res_list[lb + i] = -1;
    if (i >= nc) a.cpu_list[lb + i] = -1;
    if (i >= nd) a.delta_list[lb + i] = -1;
  }
  if (lane == 0) {
    a.topk_count[u] = nt;
    a.res_count[u] = nr;
    a.cpu_count[u] = nc;
    a.delta_count[u] = nd;
  }
}

// KIND: the digest (min/max bound or mean); SUM: the block score of a unit is the sum of its
// query heads' scores instead of their maximum.
template <int KIND, bool SUM>
__global__ void __launch_bounds__(kThreadsAll, 1) score_topk_kernel(const __grid_constant__ CUtensorMap tmD,
                                                                    const TopkArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kMaxStagesT], empty_bar[kMaxStagesT], kfull[kMaxKeyBufs], kempty[kMaxKeyBufs],
      kunit_bar[kMaxKeyBufs];
  __shared__ int stage_unit[kMaxStagesT], kunit[kMaxKeyBufs];  // unit of a stage / of a key buffer, -1 = end
  __shared__ int stage_nv[kMaxStagesT], knv[kMaxKeyBufs];       // and its valid-block count
  __shared__ int s_seq[kSeqCache];
  // dynamic shared memory: [ring (1024-aligned)][nkbuf key buffers][nsel selector-warp areas]
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint32_t* keybuf = reinterpret_cast<uint32_t*>(ring + a.stages * kStageBytesT);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kScoreWarps);
    }
    for (int i = 0; i < a.nkbuf; ++i) {
      mbar_init(&kfull[i], kScoreWarps);
      mbar_init(&kempty[i], 1);
      mbar_init(&kunit_bar[i], 1);
    }
    fence_mbar_init();
  }
  const int B = a.units / a.Hkv;
  for (int b = tid; b < min(B, kSeqCache); b += blockDim.x) s_seq[b] = a.seq_len[b];
  __syncthreads();

  if (warp == kProducer) {
    // ---------------- producer warp ------------------------------------------
    // Units are dealt out one at a time from a ticket counter, so a CTA that starts late
    // (its SM was busy) or scores a short unit simply takes more of them.  Every CTA draws
    // exactly one ticket past the last unit, and the draw of the launch's very last ticket
    // resets the counter for the next call.  A CTA whose wait has expired stops issuing
    // work but keeps drawing tickets until it draws one past the last unit, so that the
    // counter is reset all the same and the next call on the workspace starts from zero.
    if (lane != 0) return;
    prefetch_tmap(&tmD);
    const int last_ticket = a.units + (int)gridDim.x - 1;
    auto resolve = [&](int t) {
      if (t == last_ticket) *a.counters = 0;
      return t < a.units ? t : -1;
    };
    auto nvalid_of = [&](int b) {
      const int L = b < kSeqCache ? s_seq[b] : a.seq_len[b];
      return min(a.nblk_cap, (max(L, 0) + a.P - 1) / a.P);
    };
    int64_t i = 0;  // stages issued
    int st = 0;     // i % stages, kept running (no division per chunk)
    uint32_t ph = 0u;  // (i / stages) & 1
    bool q_ready = false, ok = true;
    int u = resolve(atomicAdd(a.counters, 1));
    while (u >= 0) {
      // the next ticket is drawn now and read only once this unit's stages are issued, so the
      // atomic's round trip never holds the ring up
      const int t_next = atomicAdd(a.counters, 1);
      const int nv = nvalid_of(u / a.Hkv);
      const int b = u / a.Hkv, kvh = u - b * a.Hkv;
      for (int ch = 0; ok && ch < a.nchunk; ++ch, ++i, st = st + 1 == a.stages ? 0 : st + 1, ph ^= st == 0) {
        if (!mbar_wait(&empty_bar[st], ph ^ 1u)) {
          report(a.status, SCOUT_DEV_TIMEOUT);
          ok = false;
          break;
        }
        stage_unit[st] = u;  // published by the arrive below, with the unit's valid-block count
        stage_nv[st] = nv;
        uint8_t* sp = ring + st * kStageBytesT;
        if (ch * kChunk < nv) {
          const bool with_q = ch == 0;  // the scoring warps read q on a unit's first chunk
          mbar_arrive_tx(&full_bar[st], 4 * kBoxBytes + (with_q ? a.G * kD * 2 : 0));
          const int y = u * a.nblk_cap + ch * kChunk;
#pragma unroll
          for (int bx = 0; bx < 4; ++bx) tma_load_2d(sp + bx * kBoxBytes, &tmD, bx * 64, y, &full_bar[st]);
          const __nv_bfloat16* qg = a.q + ((int64_t)b * a.Hq + (int64_t)kvh * a.G) * kD;
          if (with_q && !q_ready) {
            // started early: q is written by the kernel this launch depends on, so wait for it
            // here (the digest loads above need not); a no-op otherwise
            wait_prerequisites();
            q_ready = true;
          }
          for (int h = 0; h < (with_q ? a.G : 0); ++h)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(sp + 4 * kBoxBytes + h * kQStride * 2)),
                "l"(qg + h * kD), "r"(kD * 2), "r"(smem_u32(&full_bar[st]))
                : "memory");
        } else {
          mbar_arrive(&full_bar[st]);
        }
      }
      if (ok && a.inject == SCOUT_INJECT_ABANDON) {  // as if the next wait had expired
        report(a.status, SCOUT_DEV_TIMEOUT);
        ok = false;
      }
      u = resolve(t_next);
    }
    // every unit is handed out: a kernel that starts early after this one may take the SMs
    // this grid's CTAs leave while they finish their last units
    release_dependents();
    if (ok) {  // a stage tagged -1 ends the scoring warps' loop
      if (mbar_wait(&empty_bar[st], ph ^ 1u)) {
        stage_unit[st] = -1;
        mbar_arrive(&full_bar[st]);
        ++i;
      } else {
        report(a.status, SCOUT_DEV_TIMEOUT);
      }
    }
    for (int64_t r = 0; r < a.stages && r < i; ++r) {  // every copy lands before the CTA retires
      const int64_t last = i - 1 - r;
      if (!mbar_wait(&full_bar[last % a.stages], (uint32_t)((last / a.stages) & 1))) report(a.status, SCOUT_DEV_TIMEOUT);
    }
    return;
  }

  if (warp >= kScoreWarps) {
    // ---------------- selector warps 8..11 -----------------------------------
    // the e-th unit of this CTA sits in key buffer e % nkbuf and is selected by selector
    // warp e % nsel, so up to nsel units are selected at once; its id arrives when its
    // scoring starts, so the residency bits load while it is scored
    const int sw_i = warp - kScoreWarps;
    if (sw_i >= a.nsel) return;
    uint32_t* area = keybuf + a.nkbuf * align4(a.nblk_cap) + sw_i * selwarp_words(a.words);
    const SelWarp sw = selwarp_at(area, a.words);
    for (int e = sw_i;; e += a.nsel) {
      const int kb = e % a.nkbuf;
      if (!mbar_wait(&kunit_bar[kb], (uint32_t)(e / a.nkbuf) & 1u)) {
        if (lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
        return;
      }
      const int u = kunit[kb], nvalid = knv[kb];
      if (u < 0) return;
      uint32_t* keys = keybuf + kb * align4(a.nblk_cap);
      prefetch_unit(a, u, sw, lane);  // overlaps the scoring of u
      if (!mbar_wait(&kfull[kb], (uint32_t)(e / a.nkbuf) & 1u) && lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
      select_unit(a, u, keys, nvalid, sw, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&kempty[kb]);  // the key buffer may be refilled
    }
    return;
  }

  // ---------------- scoring warps 0..7 -----------------------------------------
  const int g = lane >> 2, t = lane & 3;
  const TileOfs tofs = KIND == SCOUT_DIGEST_MINMAX ? minmax_offsets(warp * 16, lane) : mean_offsets(warp * 16, lane);
  int ucur = -1, kb = 0, e = -1, ch = 0, nvalid = 0;
  uint32_t bmm[16][2], bme[8][2];
  // stage st of the ring, phase ph, advanced after every chunk (no division per chunk)
  for (int st = 0, ph = 0;; st = st + 1 == a.stages ? 0 : st + 1, ph ^= st == 0) {
    const bool landed = mbar_wait_n(&full_bar[st], (uint32_t)ph, a.score_wait);
    if (!landed && lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
    const int u = landed ? stage_unit[st] : -1;
    if (u < 0) break;
    const uint8_t* sp = ring + st * kStageBytesT;
    if (u != ucur) {  // the unit's first chunk: take its key buffer and read its query group
      ucur = u;
      ch = 0;
      ++e;
      kb = e % a.nkbuf;
      nvalid = stage_nv[st];
      if (!mbar_wait(&kempty[kb], ((uint32_t)(e / a.nkbuf) & 1u) ^ 1u) && lane == 0)
        report(a.status, SCOUT_DEV_TIMEOUT);
      if (warp == 0 && lane == 0) {
        kunit[kb] = u;
        knv[kb] = nvalid;
        mbar_arrive(&kunit_bar[kb]);
      }
      if (nvalid > 0) {
        const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(sp + 4 * kBoxBytes);
        if (KIND == SCOUT_DIGEST_MINMAX) {
          minmax_b_frag(qs, a.G, lane, bmm);
        } else {
          mean_b_frag(qs, a.G, lane, bme);
        }
      }
    }
    const int j0 = ch * kChunk + warp * 16;
    if (j0 < a.nblk_cap) {
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      if (j0 < nvalid) score_tile<KIND>(smem_u32(sp), tofs, bmm, bme, c);
      // pool over the heads of the group (columns 2t, 2t+1 < G), then across t; for the sum the
      // order is ((h0 + h1) + (h2 + h3)) + ((h4 + h5) + (h6 + h7)), the same on every lane
      const float ninf = -INFINITY;
      float m0, m1;
      if (SUM) {
        m0 = (2 * t < a.G ? c[0] : 0.f) + (2 * t + 1 < a.G ? c[1] : 0.f);
        m1 = (2 * t < a.G ? c[2] : 0.f) + (2 * t + 1 < a.G ? c[3] : 0.f);
        m0 += __shfl_xor_sync(0xffffffffu, m0, 1);
        m0 += __shfl_xor_sync(0xffffffffu, m0, 2);
        m1 += __shfl_xor_sync(0xffffffffu, m1, 1);
        m1 += __shfl_xor_sync(0xffffffffu, m1, 2);
      } else {
        m0 = fmaxf(2 * t < a.G ? c[0] : ninf, 2 * t + 1 < a.G ? c[1] : ninf);
        m1 = fmaxf(2 * t < a.G ? c[2] : ninf, 2 * t + 1 < a.G ? c[3] : ninf);
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
      }
      if (t == 0) {
        const int r0 = j0 + g, r1 = j0 + g + 8;
        uint32_t* keys = keybuf + kb * align4(a.nblk_cap);
        if (r0 < nvalid) keys[r0] = score_key(m0);
        if (r1 < nvalid) keys[r1] = score_key(m1);
        if (a.user_scores) {
          float* scu = a.scores + (int64_t)u * a.nblk_cap;
          if (r0 < a.nblk_cap) scu[r0] = r0 < nvalid ? m0 : ninf;
          if (r1 < a.nblk_cap) scu[r1] = r1 < nvalid ? m1 : ninf;
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty_bar[st]);
      if (ch == a.nchunk - 1) mbar_arrive(&kfull[kb]);  // this warp's keys of u are in
    }
    ++ch;
  }
  // no more units: an id of -1 in the next key buffer of every selector warp ends its loop
  for (int j = 0; j < a.nsel; ++j) {
    const int e2 = e + 1 + j, kb2 = e2 % a.nkbuf;
    if (!mbar_wait(&kempty[kb2], ((uint32_t)(e2 / a.nkbuf) & 1u) ^ 1u) && lane == 0)
      report(a.status, SCOUT_DEV_TIMEOUT);
    if (warp == 0 && lane == 0) {
      kunit[kb2] = -1;
      mbar_arrive(&kunit_bar[kb2]);
    }
  }
}

inline size_t counters_bytes(int64_t units) { return (size_t)((units * 4 + 255) / 256 * 256); }

}  // namespace
}  // namespace scout

extern "C" size_t scout_score_topk_workspace_bytes(int B, int Hkv, int nblk_cap) {
  if (B <= 0 || Hkv <= 0 || nblk_cap <= 0) return 0;
  const int64_t units = (int64_t)B * Hkv;
  return scout::counters_bytes(units);  // the unit ticket counter (room for one word per unit)
}

namespace scout {
namespace {

// Every host-side check of scout_score_topk except the workspace's: SCOUT_OK or the error.
int check_topk_args(int kind, const void* q, const void* digest, const int32_t* seq_len,
                    const uint32_t* resident_bits, const int32_t* prev_cpu_list, const int32_t* prev_cpu_count,
                    int B, int Hq, int Hkv, int D, int P, int nblk_cap, int k, const int32_t* topk_idx,
                    const int32_t* topk_count, const int32_t* res_list, const int32_t* res_count,
                    const int32_t* cpu_list, const int32_t* cpu_count, const int32_t* delta_list,
                    const int32_t* delta_count, const scout_launch* launch) {
  if (q == nullptr || digest == nullptr || seq_len == nullptr || resident_bits == nullptr || topk_idx == nullptr ||
      topk_count == nullptr || res_list == nullptr || res_count == nullptr || cpu_list == nullptr ||
      cpu_count == nullptr || delta_list == nullptr || delta_count == nullptr)
    return SCOUT_ERR_INVALID_ARG;
  if ((prev_cpu_list == nullptr) != (prev_cpu_count == nullptr)) return SCOUT_ERR_INVALID_ARG;
  if (launch != nullptr && (launch->max_ctas < 0 || launch->inject < SCOUT_INJECT_NONE ||
                            launch->inject > SCOUT_INJECT_ABANDON))
    return SCOUT_ERR_INVALID_ARG;
  kind &= ~SCOUT_POOL_SUM;
  if (kind != SCOUT_DIGEST_MINMAX && kind != SCOUT_DIGEST_MEAN) return SCOUT_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || nblk_cap <= 0 || k <= 0) return SCOUT_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  const int64_t units = (int64_t)B * Hkv;
  if (D != kD || !valid_P(P) || G > kMaxG || nblk_cap > kMaxNblk || units * nblk_cap > 0x7fffffffLL ||
      !aligned16(digest) || !aligned16(q))
    return SCOUT_ERR_UNSUPPORTED;
  return SCOUT_OK;
}

// Poll limit of the scoring warps' stage waits under SCOUT_INJECT_ABANDON: long enough for
// any copy that was issued to land, short enough that the test's expired wait ends quickly.
constexpr uint32_t kInjectWaitLimit = 1u << 15;

}  // namespace
}  // namespace scout

namespace scout {
namespace {
// scout_score_topk; with zero_counter set, the workspace's counter bytes are zeroed on the
// stream after every host-side check has passed, just before the launch.
int score_topk_entry(int kind, const void* q, const void* digest, const int32_t* seq_len,
                     const uint32_t* resident_bits, const int32_t* prev_cpu_list, const int32_t* prev_cpu_count, int B,
                     int Hq, int Hkv, int D, int P, int nblk_cap, int k, float* scores, int32_t* topk_idx,
                     int32_t* topk_count, int32_t* res_list, int32_t* res_count, int32_t* cpu_list,
                     int32_t* cpu_count, int32_t* delta_list, int32_t* delta_count, void* workspace,
                     size_t workspace_bytes, int32_t* dev_status, const scout_launch* launch, cudaStream_t stream,
                     bool zero_counter) {
  const int rc = check_topk_args(kind, q, digest, seq_len, resident_bits, prev_cpu_list, prev_cpu_count, B, Hq, Hkv,
                                 D, P, nblk_cap, k, topk_idx, topk_count, res_list, res_count, cpu_list, cpu_count,
                                 delta_list, delta_count, launch);
  if (rc != SCOUT_OK) return rc;
  if (workspace == nullptr || workspace_bytes < scout_score_topk_workspace_bytes(B, Hkv, nblk_cap))
    return SCOUT_ERR_WORKSPACE;
  const bool sum_pool = (kind & SCOUT_POOL_SUM) != 0;
  kind &= ~SCOUT_POOL_SUM;
  const int G = Hq / Hkv;
  const int64_t units = (int64_t)B * Hkv;
  TopkArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.digest = static_cast<const uint8_t*>(digest);
  a.seq_len = seq_len;
  a.resident_bits = resident_bits;
  a.prev_list = prev_cpu_list;
  a.prev_count = prev_cpu_count;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.P = P;
  a.nblk_cap = nblk_cap;
  a.k = k;
  a.words = (nblk_cap + 31) / 32;
  a.nchunk = (nblk_cap + kChunk - 1) / kChunk;
  a.units = (int)units;
  a.counters = static_cast<int32_t*>(workspace);
  a.status = dev_status;
  a.inject = launch != nullptr ? launch->inject : SCOUT_INJECT_NONE;
  a.score_wait = a.inject == SCOUT_INJECT_ABANDON ? kInjectWaitLimit : kWaitLimit;
  a.user_scores = scores != nullptr;
  a.scores = scores;
  a.topk_idx = topk_idx;
  a.topk_count = topk_count;
  a.res_list = res_list;
  a.res_count = res_count;
  a.cpu_list = cpu_list;
  a.cpu_count = cpu_count;
  a.delta_list = delta_list;
  a.delta_count = delta_count;
  // the digest as a 2-D bf16 tensor [units * nblk_cap rows][256 columns] (512-byte rows
  // for both kinds); 128-row x 64-column boxes with the 128-byte swizzle
  CUtensorMap tmD;
  {
    const cuuint64_t dims[2] = {256, (cuuint64_t)units * nblk_cap};
    const cuuint64_t strides[1] = {512};
    const cuuint32_t box[2] = {64, (cuuint32_t)kChunk};
    const cuuint32_t estr[2] = {1, 1};
    if (encode_tiled(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(digest), dims, strides, box, estr,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return SCOUT_ERR_UNSUPPORTED;
  }
  // per-block limit 232448 bytes (227 KiB) covers static (< 2 KiB here) and dynamic shared
  // memory: the most ring stages, then the most key buffers (at least two) that fit
  const size_t avail = 232448 - 2048 - 1024;
  const size_t kbuf_bytes = (size_t)align4(nblk_cap) * 4, selw_bytes = (size_t)selwarp_words(a.words) * 4;
  auto need = [&](int stages, int nkbuf) {
    return (size_t)stages * kStageBytesT + nkbuf * kbuf_bytes + min(kSelWarps, nkbuf - 1) * selw_bytes;
  };
  a.stages = 0;
  for (int st = kMaxStagesT; st >= 1 && a.stages == 0; --st)
    for (int nk = kMaxKeyBufs; nk >= 2; --nk)
      if (need(st, nk) <= avail) {
        a.stages = st;
        a.nkbuf = nk;
        break;
      }
  if (a.stages == 0) return SCOUT_ERR_UNSUPPORTED;
  a.nsel = min(kSelWarps, a.nkbuf - 1);
  const size_t smem = 1024 + need(a.stages, a.nkbuf);
  auto kern = kind == SCOUT_DIGEST_MINMAX
                  ? (sum_pool ? score_topk_kernel<SCOUT_DIGEST_MINMAX, true> : score_topk_kernel<SCOUT_DIGEST_MINMAX, false>)
                  : (sum_pool ? score_topk_kernel<SCOUT_DIGEST_MEAN, true> : score_topk_kernel<SCOUT_DIGEST_MEAN, false>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return SCOUT_ERR_CUDA;
  // Default grid: the fewest CTAs that still take ceil(units / SMs) units each, so that the last
  // round of units does not leave most SMs idle while a few stream on (320 units on 152 SMs: 107
  // CTAs of three units rather than 152 CTAs of which 16 take a third).  A cap is taken as given.
  int cap = launch != nullptr ? launch->max_ctas : 0;
  if (cap <= 0) {
    const int64_t sms = sm_count(), rounds = (units + sms - 1) / sms;
    cap = (int)((units + rounds - 1) / rounds);
  }
  const int grid = (int)(units < (int64_t)cap ? units : (int64_t)cap);  // <= one CTA per unit
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreadsAll);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = early_start_attrs(launch, attr, 0);
  if (zero_counter && cudaMemsetAsync(workspace, 0, counters_bytes(units), stream) != cudaSuccess)
    return SCOUT_ERR_CUDA;
  if (cudaLaunchKernelEx(&cfg, kern, tmD, a) != cudaSuccess) return SCOUT_ERR_CUDA;
  return launch_status();
}
}  // namespace
}  // namespace scout

extern "C" int scout_score_topk(int kind, const void* q, const void* digest, const int32_t* seq_len,
                                const uint32_t* resident_bits, const int32_t* prev_cpu_list,
                                const int32_t* prev_cpu_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap,
                                int k, float* scores, int32_t* topk_idx, int32_t* topk_count, int32_t* res_list,
                                int32_t* res_count, int32_t* cpu_list, int32_t* cpu_count, int32_t* delta_list,
                                int32_t* delta_count, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                const scout_launch* launch, cudaStream_t stream) {
  return scout::score_topk_entry(kind, q, digest, seq_len, resident_bits, prev_cpu_list, prev_cpu_count, B, Hq, Hkv,
                                 D, P, nblk_cap, k, scores, topk_idx, topk_count, res_list, res_count, cpu_list,
                                 cpu_count, delta_list, delta_count, workspace, workspace_bytes, dev_status, launch,
                                 stream, false);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of scout_score_topk.
//
// Some callers cannot allocate device memory at the point where they select
// blocks: engines that reserve all GPU memory in one pool at start-up and forbid
// later cudaMalloc calls (a cudaMalloc can stall other streams and fragment the
// pool), or hosts that load this library as a plugin and hand it no allocator.
// For them the scratch lives in one file-scope device array of fixed size that
// every GPU loading the library keeps until the process exits.
// ---------------------------------------------------------------------------
namespace scout {
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB, sized as a workspace of B * Hkv <= 1,048,576 units
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kNoAllocMaxDevices] = {};

// Device address of g_topk_scratch on the current device (the host-side symbol is only a
// stand-in and must never reach a kernel).  Looked up afresh whenever `stream` is not being
// captured, so that a cudaDeviceReset (after which the module, and the array, are loaded
// anew) cannot leave a stale address behind; during a capture the address found by the last
// call outside one is used, since the lookup may load the module.
int scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SCOUT_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return SCOUT_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SCOUT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr) return SCOUT_ERR_CUDA;
    g_scratch_addr[dev] = p;
  } else if (g_scratch_addr[dev] == nullptr) {
    return SCOUT_ERR_CUDA;  // never called on this device outside a capture
  }
  *out = g_scratch_addr[dev];
  return SCOUT_OK;
}

}  // namespace
}  // namespace scout

extern "C" size_t scout_score_topk_noalloc_max_bytes(void) { return scout::kNoAllocScratchBytes; }

extern "C" int scout_score_topk_noalloc(int kind, const void* q, const void* digest, const int32_t* seq_len,
                                        const uint32_t* resident_bits, const int32_t* prev_cpu_list,
                                        const int32_t* prev_cpu_count, int B, int Hq, int Hkv, int D, int P,
                                        int nblk_cap, int k, float* scores, int32_t* topk_idx, int32_t* topk_count,
                                        int32_t* res_list, int32_t* res_count, int32_t* cpu_list, int32_t* cpu_count,
                                        int32_t* delta_list, int32_t* delta_count, int32_t* dev_status,
                                        cudaStream_t stream) {
  using namespace scout;
  // every argument is checked before the shared array is touched
  const int rc = check_topk_args(kind, q, digest, seq_len, resident_bits, prev_cpu_list, prev_cpu_count, B, Hq, Hkv,
                                 D, P, nblk_cap, k, topk_idx, topk_count, res_list, res_count, cpu_list, cpu_count,
                                 delta_list, delta_count, nullptr);
  if (rc != SCOUT_OK) return rc;
  if (scout_score_topk_workspace_bytes(B, Hkv, nblk_cap) > kNoAllocScratchBytes) return SCOUT_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int ra = scratch_address(stream, &scratch);
  if (ra != SCOUT_OK) return ra;
  // the array keeps whatever the previous call left: its counter is zeroed on the stream once
  // the remaining checks have passed, just before the launch
  return score_topk_entry(kind, q, digest, seq_len, resident_bits, prev_cpu_list, prev_cpu_count, B, Hq, Hkv, D, P,
                          nblk_cap, k, scores, topk_idx, topk_count, res_list, res_count, cpu_list, cpu_count,
                          delta_list, delta_count, scratch, kNoAllocScratchBytes, dev_status, nullptr, stream, true);
}
