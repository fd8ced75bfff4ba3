// scout_sparse_attn: split-K paged GQA decode attention over the resident
// selected blocks.  ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1
// (A_gpu = GPUATTN(Q, B_gpu)): the GPU attends the top-k blocks in its memory.
//
// Work partition (balanced over the SMs): the resident selected blocks of all
// units form one list of N = sum_u res_count[u] blocks.  CTA c of Gp = min(grid,
// N) takes the contiguous range [c N / Gp, (c+1) N / Gp).  A unit that falls
// inside one range is finished by that CTA; a unit split over several CTAs is
// finished by the last of them to arrive (self-resetting counter), which merges
// the per-CTA partials by their LSE.
//
// Inside a CTA: warp 4 lane 0 streams K and V pages into a ring of shared-memory
// stages with TMA (cp.async.bulk.tensor, 128-byte swizzle) and mbarriers; the
// four consumer warps take blocks round-robin, run S = Q K^T and O += P V on the
// tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate; P is split into a
// bf16 high and low part so the probabilities keep ~16 significant bits) and
// keep an online softmax per warp, combined through shared memory at the end of
// each unit segment.
#include "common.cuh"

namespace scout {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxUnits = 4096;
constexpr int kMaxGrid = 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int P>
struct Cfg {
  static constexpr int kStages = P == 16 ? 8 : 4;
  static constexpr int kHalfBytes = P * 128;        // one 64-column half of a page
  static constexpr int kStageBytes = 4 * kHalfBytes; // K (2 halves) + V (2 halves)
  static constexpr int kRingBytes = kStages * kStageBytes;
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
  float* O_part;
  float* lse_part;
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

// Slot of block j of unit u, or -1 when it is out of range (skipped, reported).
__device__ __forceinline__ int64_t block_slot(const AttnArgs& a, int u, int j, int P, int* ntok) {
  const int b = u / a.Hkv;
  if (j < 0 || j >= a.nblk_cap) return -1;
  const int nv = min(P, a.seq_len[b] - j * P);
  if (nv <= 0) return -1;
  const int32_t s = a.page_table[(int64_t)u * a.nblk_cap + j];
  if (s < 0 || s >= a.n_slots) return -1;
  *ntok = nv;
  return s;
}

// Row address (shared::cta) of token r, 16-byte chunk C (dims 8C..8C+7) in a
// page stored as two 64-column halves with the 128-byte TMA swizzle.
template <int P>
__device__ __forceinline__ uint32_t page_addr(uint32_t base, int r, int C) {
  return base + (uint32_t)((C >> 3) * Cfg<P>::kHalfBytes + r * 128 + ((((C & 7) ^ (r & 7))) << 4));
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

struct WarpState {
  float m;       // running max of scaled scores (log2 units), row g
  float l;       // running sum of exp2(s - m), this lane's columns only
  float o[16][4];
};

// One page: S = Q K^T, online softmax, O += P V.
template <int P>
__device__ __forceinline__ void attend_page(uint32_t kbase, uint32_t vbase, int ntok, const uint32_t (&qa)[8][2],
                                            float scale_log2, WarpState& st, int lane) {
  constexpr int NT = P / 8;
  const int t = lane & 3;
  float s[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    const int r = nt * 8 + (lane & 7);
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(page_addr<P>(kbase, r, 4 * kp + (lane >> 3)), b0, b1, b2, b3);
      mma_bf16(s[nt], qa[2 * kp][0], 0u, qa[2 * kp][1], 0u, b0, b1);
      mma_bf16(s[nt], qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u, b2, b3);
    }
  }
  float bmax = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tok = nt * 8 + 2 * t + e;
      s[nt][e] = tok < ntok ? s[nt][e] * scale_log2 : -INFINITY;
      bmax = fmaxf(bmax, s[nt][e]);
    }
  }
  bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 1));
  bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 2));
  const float m_new = fmaxf(st.m, bmax);
  const float alpha = exp2f(st.m - m_new);  // 0 on the first page (m = -inf)
  st.m = m_new;
  float psum = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    s[nt][0] = exp2f(s[nt][0] - m_new);
    s[nt][1] = exp2f(s[nt][1] - m_new);
    psum += s[nt][0] + s[nt][1];
  }
  st.l = st.l * alpha + psum;
#pragma unroll
  for (int d = 0; d < 16; ++d) {
    st.o[d][0] *= alpha;
    st.o[d][1] *= alpha;
  }
#pragma unroll
  for (int kk = 0; kk < P / 16; ++kk) {
    const uint32_t h0 = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
    const uint32_t h2 = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
    const uint32_t l0 = pack_bf16(s[2 * kk][0] - bf16_lo(h0), s[2 * kk][1] - bf16_hi(h0));
    const uint32_t l2 = pack_bf16(s[2 * kk + 1][0] - bf16_lo(h2), s[2 * kk + 1][1] - bf16_hi(h2));
    const int r = kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
    for (int dp = 0; dp < 8; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(page_addr<P>(vbase, r, 2 * dp + (lane >> 4)), b0, b1, b2, b3);
      mma_bf16(st.o[2 * dp], h0, 0u, h2, 0u, b0, b1);
      mma_bf16(st.o[2 * dp], l0, 0u, l2, 0u, b0, b1);
      mma_bf16(st.o[2 * dp + 1], h0, 0u, h2, 0u, b2, b3);
      mma_bf16(st.o[2 * dp + 1], l0, 0u, l2, 0u, b2, b3);
    }
  }
}

template <int P>
__global__ void __launch_bounds__(kThreads) sparse_attn_kernel(const __grid_constant__ CUtensorMap tmK,
                                                               const __grid_constant__ CUtensorMap tmV,
                                                               const AttnArgs a) {
  using C = Cfg<P>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[C::kStages], empty_bar[C::kStages];
  __shared__ float cm[kConsumerWarps][kMaxG], cl[kConsumerWarps][kMaxG];
  __shared__ int wtot[kThreads / 32];
  __shared__ int s_last;

  // dynamic shared memory: [ring (1024-aligned)][combine O][unit prefix]
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  float* co = reinterpret_cast<float*>(ring + C::kRingBytes);          // [4][kMaxG][kD]
  int* prefix = reinterpret_cast<int*>(co + kConsumerWarps * kMaxG * kD);  // [units + 1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  // exclusive prefix of the clamped resident counts over all units
  {
    const int per = (a.units + kThreads - 1) / kThreads;
    const int lo = min(a.units, tid * per), hi = min(a.units, lo + per);
    int sum = 0;
    for (int u = lo; u < hi; ++u) sum += min(max(a.res_count[u], 0), a.k);
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
      prefix[u] = run;
      run += min(max(a.res_count[u], 0), a.k);
    }
    if (tid == kThreads - 1) prefix[a.units] = run;
    __syncthreads();
  }
  const int64_t N = prefix[a.units];
  const int Gp = (int)min((int64_t)((int64_t)gridDim.x), (int64_t)(N));
  const int c = blockIdx.x;

  if (warp == kConsumerWarps) {
    // ---------------- producer: one thread streams pages -----------------
    if (lane != 0 || c >= Gp) return;
    const int64_t start = range_start(c, N, Gp), end = range_start(c + 1, N, Gp);
    int u = 0;
    {
      int lo = 0, hi = a.units - 1;  // last unit with prefix[u] <= start
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= start) lo = mid; else hi = mid - 1;
      }
      u = lo;
    }
    uint32_t i = 0;
    bool ok = true;
    for (int64_t pos = start; pos < end && ok; ++u) {
      const int64_t seg_hi = min((int64_t)(end), (int64_t)(prefix[u + 1]));
      for (; pos < seg_hi; ++pos, ++i) {
        const int stage = (int)(i % C::kStages);
        if (!mbar_wait(&empty_bar[stage], ((i / C::kStages) & 1u) ^ 1u)) {
          report(a.status, SCOUT_DEV_TIMEOUT);
          ok = false;
          break;
        }
        const int j = a.res_list[(int64_t)u * a.k + (pos - prefix[u])];
        int ntok = 0;
        const int64_t slot = block_slot(a, u, j, P, &ntok);
        if (slot < 0) {
          report(a.status, SCOUT_DEV_BAD_INDEX);
          mbar_arrive(&full_bar[stage]);
          continue;
        }
        uint8_t* st = ring + stage * C::kStageBytes;
        mbar_arrive_tx(&full_bar[stage], C::kStageBytes);
        const int y = (int)(slot * P);
        tma_load_2d(st, &tmK, 0, y, &full_bar[stage]);
        tma_load_2d(st + C::kHalfBytes, &tmK, 64, y, &full_bar[stage]);
        tma_load_2d(st + 2 * C::kHalfBytes, &tmV, 0, y, &full_bar[stage]);
        tma_load_2d(st + 3 * C::kHalfBytes, &tmV, 64, y, &full_bar[stage]);
      }
    }
    // drain: wait until every copy issued into a stage has landed
    for (uint32_t r = 0; r < C::kStages && r < i; ++r) {
      const uint32_t last = i - 1 - r;
      if (!mbar_wait(&full_bar[last % C::kStages], (last / C::kStages) & 1u)) report(a.status, SCOUT_DEV_TIMEOUT);
    }
    return;
  }

  // ---------------- consumers (warps 0..3) ---------------------------------
  const int g = lane >> 2, t = lane & 3;
  // units with no resident selected block: O = 0, lse = -inf
  for (int u = c; u < a.units; u += gridDim.x) {
    if (prefix[u + 1] != prefix[u]) continue;
    for (int idx = tid; idx < a.G * kD; idx += kConsumerWarps * 32) a.O_part[(int64_t)u * a.G * kD + idx] = 0.f;
    if (tid < a.G) a.lse_part[(int64_t)u * a.G + tid] = -INFINITY;
  }
  if (c >= Gp) return;
  const int64_t start = range_start(c, N, Gp), end = range_start(c + 1, N, Gp);
  int u0 = 0;
  {
    int lo = 0, hi = a.units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= start) lo = mid; else hi = mid - 1;
    }
    u0 = lo;
  }
  const uint32_t ring_s = smem_u32(ring);
  uint32_t i = 0;
  for (int64_t pos = start, u = u0; pos < end; ++u) {
    const int64_t seg_lo = pos, seg_hi = min((int64_t)(end), (int64_t)(prefix[u + 1]));
    if (seg_hi <= seg_lo) continue;
    const int b = (int)(u / a.Hkv), kvh = (int)(u - (int64_t)b * a.Hkv);
    uint32_t qa[8][2];
    const __nv_bfloat16* qrow = a.q + ((int64_t)b * a.Hq + (int64_t)kvh * a.G + g) * kD;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = g < a.G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * t) : 0u;
      qa[ks][1] = g < a.G ? *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * t) : 0u;
    }
    WarpState st;
    st.m = -INFINITY;
    st.l = 0.f;
#pragma unroll
    for (int d = 0; d < 16; ++d) st.o[d][0] = st.o[d][1] = st.o[d][2] = st.o[d][3] = 0.f;
    for (int64_t p = seg_lo; p < seg_hi; ++p, ++i) {
      if ((int)(i % kConsumerWarps) != warp) continue;
      const int stage = (int)(i % C::kStages);
      if (!mbar_wait(&full_bar[stage], (i / C::kStages) & 1u)) {
        if (lane == 0) report(a.status, SCOUT_DEV_TIMEOUT);
      } else {
        const int j = a.res_list[u * a.k + (p - prefix[u])];
        int ntok = 0;
        if (block_slot(a, (int)u, j, P, &ntok) >= 0) {
          const uint32_t kb = ring_s + stage * C::kStageBytes;
          attend_page<P>(kb, kb + 2 * C::kHalfBytes, ntok, qa, a.scale_log2, st, lane);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[stage]);
    }
    pos = seg_hi;

    // combine the four warps of this CTA
    float lsum = st.l + __shfl_xor_sync(0xffffffffu, st.l, 1);
    lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
    if (g < a.G) {
      if (t == 0) {
        cm[warp][g] = st.m;
        cl[warp][g] = lsum;
      }
      float* dst = co + (warp * kMaxG + g) * kD;
#pragma unroll
      for (int d = 0; d < 16; ++d) {
        dst[d * 8 + 2 * t] = st.o[d][0];
        dst[d * 8 + 2 * t + 1] = st.o[d][1];
      }
    }
    consumer_sync();
    const bool whole = seg_lo == prefix[u] && seg_hi == prefix[u + 1];
    const int which = prefix[u] <= start ? 0 : 1;
    for (int idx = tid; idx < a.G * kD; idx += kConsumerWarps * 32) {
      const int h = idx / kD, d = idx - h * kD;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cm[w][h]);
      float L = 0.f, acc = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float f = exp2f(cm[w][h] - M);
          L += cl[w][h] * f;
          acc += co[(w * kMaxG + h) * kD + d] * f;
        }
      }
      const float O = L > 0.f ? acc / L : 0.f;
      const float lse = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      if (whole) {
        a.O_part[(u * a.G + h) * kD + d] = O;
        if (d == 0) a.lse_part[u * a.G + h] = lse;
      } else {
        const int64_t sl = (int64_t)c * 2 + which;
        a.slot_O[(sl * kMaxG + h) * kD + d] = O;
        if (d == 0) a.slot_lse[sl * kMaxG + h] = lse;
      }
    }
    if (!whole) {
      __threadfence();
      consumer_sync();
      const int c0 = cta_of(prefix[u], N, Gp), c1 = cta_of(prefix[u + 1] - 1, N, Gp);
      if (tid == 0) s_last = atomicAdd(&a.counters[u], 1) == c1 - c0;
      consumer_sync();
      if (s_last) {
        __threadfence();
        for (int idx = tid; idx < a.G * kD; idx += kConsumerWarps * 32) {
          const int h = idx / kD, d = idx - h * kD;
          float M = -INFINITY;
          for (int cc = c0; cc <= c1; ++cc) {
            const int64_t sl = (int64_t)cc * 2 + (prefix[u] <= range_start(cc, N, Gp) ? 0 : 1);
            M = fmaxf(M, __ldcg(a.slot_lse + sl * kMaxG + h));
          }
          float L = 0.f, acc = 0.f;
          if (M != -INFINITY) {
            for (int cc = c0; cc <= c1; ++cc) {
              const int64_t sl = (int64_t)cc * 2 + (prefix[u] <= range_start(cc, N, Gp) ? 0 : 1);
              const float f = expf(__ldcg(a.slot_lse + sl * kMaxG + h) - M);
              L += f;
              acc += f * __ldcg(a.slot_O + (sl * kMaxG + h) * kD + d);
            }
          }
          a.O_part[(u * a.G + h) * kD + d] = L > 0.f ? acc / L : 0.f;
          if (d == 0) a.lse_part[u * a.G + h] = L > 0.f ? M + logf(L) : -INFINITY;
        }
        if (tid == 0) a.counters[u] = 0;  // ready for the next call
      }
    }
    consumer_sync();  // the combine scratch is reused by the next segment
  }
}

inline size_t counters_bytes(int64_t units) { return (size_t)((units * 4 + 255) / 256 * 256); }
constexpr size_t kSlotLseBytes = (size_t)kMaxGrid * 2 * kMaxG * sizeof(float);
constexpr size_t kSlotOBytes = (size_t)kMaxGrid * 2 * kMaxG * kD * sizeof(float);

template <int P>
size_t dyn_smem(int units) {
  return 1024 + Cfg<P>::kRingBytes + (size_t)kConsumerWarps * kMaxG * kD * sizeof(float) + (size_t)(units + 1) * 4;
}

bool make_page_map(CUtensorMap* map, const void* pool, int64_t n_slots, int P) {
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)(n_slots * P)};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)P};
  const cuuint32_t estr[2] = {1, 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
                      CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS;
}

template <int P>
int launch_attn(const void* K_pool, const void* V_pool, const AttnArgs& a, cudaStream_t stream) {
  CUtensorMap tmK, tmV;
  if (!make_page_map(&tmK, K_pool, a.n_slots, P) || !make_page_map(&tmV, V_pool, a.n_slots, P))
    return SCOUT_ERR_UNSUPPORTED;
  const size_t smem = dyn_smem<P>(a.units);
  if (cudaFuncSetAttribute(sparse_attn_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SCOUT_ERR_CUDA;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sparse_attn_kernel<P>, kThreads, smem) != cudaSuccess ||
      occ < 1)
    return SCOUT_ERR_CUDA;
  const int grid = min(kMaxGrid, sm_count() * occ);
  sparse_attn_kernel<P><<<grid, kThreads, smem, stream>>>(tmK, tmV, a);
  return launch_status();
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
                                 int32_t* dev_status, cudaStream_t stream) {
  using namespace scout;
  if (q == nullptr || K_pool == nullptr || V_pool == nullptr || page_table == nullptr || seq_len == nullptr ||
      res_list == nullptr || res_count == nullptr || O_part == nullptr || lse_part == nullptr)
    return SCOUT_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || n_slots <= 0 || nblk_cap <= 0 || k <= 0 ||
      !(scale > 0.f))
    return SCOUT_ERR_INVALID_ARG;
  const int64_t units = (int64_t)B * Hkv;
  const int G = Hq / Hkv;
  if (D != kD || !valid_P(P) || G > kMaxG || units > kMaxUnits || !aligned16(K_pool) || !aligned16(V_pool) ||
      (reinterpret_cast<uintptr_t>(q) & 3u) || n_slots * P > (int64_t)0x7fffffff)
    return SCOUT_ERR_UNSUPPORTED;
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
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.counters = reinterpret_cast<int32_t*>(ws);
  a.slot_lse = reinterpret_cast<float*>(ws + counters_bytes(units));
  a.slot_O = reinterpret_cast<float*>(ws + counters_bytes(units) + kSlotLseBytes);
  a.status = dev_status;
  switch (P) {
    case 16: return launch_attn<16>(K_pool, V_pool, a, stream);
    case 32: return launch_attn<32>(K_pool, V_pool, a, stream);
    default: return launch_attn<64>(K_pool, V_pool, a, stream);
  }
}
