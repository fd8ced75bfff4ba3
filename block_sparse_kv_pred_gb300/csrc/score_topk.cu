// scout_score_topk: digest scoring, per-unit top-k, residency split, CPU work list.
// ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1: B_pred = TopK(q K_digest^T),
// B_cpu = B_pred \ B_gpu.
//
// Phase 1 (every CTA): a chunk of 128 blocks of one unit is scored on the tensor
// cores.  The score is a dot product over 256 (min/max) or 3 x 128 (mean, fp32
// split exactly into three bf16 terms) digest values, so each warp computes a
// 16-block x 8-head tile with mma.sync (exact bf16 products, fp32 sums).  The k
// order inside the MMA is permuted so that every lane loads 16 contiguous digest
// bytes per instruction; the query fragment uses the same permutation.
// Phase 2 (last CTA of each unit, found with a self-resetting counter): radix
// select of the k-th key, then ordered compaction into the four lists.
#include "common.cuh"

namespace scout {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = kWarps * 16;  // blocks scored per CTA

__device__ __forceinline__ uint32_t trunc_bf16(float x) { return __float_as_uint(x) & 0xFFFF0000u; }

// Orderable key of an fp32 score: larger score -> larger key; -0 and +0 equal.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t b = __float_as_uint(s == 0.f ? 0.f : s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// q fragment (B operand) for the min/max kind.  k-step s of lane (g, t) covers
// digest chunk q = (s / 2) * 4 + t (8 values); part q / 16 is min (pairs with
// q-) or max (pairs with q+); channel (q % 16) * 8 + (s % 2) * 4 + {0..3}.
__device__ __forceinline__ void minmax_b_frag(const __nv_bfloat16* qs, int G, int lane, uint32_t (&bf)[16][2]) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int s = 0; s < 16; ++s) {
    const int qc = (s >> 1) * 4 + t;
    const bool is_max = qc >= 16;
    const int ch = (qc & 15) * 8 + (s & 1) * 4;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float x = g < G ? __bfloat162float(qs[g * kD + ch + e]) : 0.f;
      v[e] = is_max ? fmaxf(x, 0.f) : fminf(x, 0.f);
    }
    bf[s][0] = pack_bf16(v[0], v[1]);
    bf[s][1] = pack_bf16(v[2], v[3]);
  }
}

// q fragment for the mean kind: load i of lane t covers channels i*16 + t*4 + {0..3}.
__device__ __forceinline__ void mean_b_frag(const __nv_bfloat16* qs, int G, int lane, uint32_t (&bf)[8][2]) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int ch = i * 16 + t * 4;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = g < G ? __bfloat162float(qs[g * kD + ch + e]) : 0.f;
    bf[i][0] = pack_bf16(v[0], v[1]);
    bf[i][1] = pack_bf16(v[2], v[3]);
  }
}

// Scores of rows j0 + g and j0 + g + 8 for heads 2t, 2t+1 (c[0..3]).
template <int KIND>
__device__ __forceinline__ void score_tile(const uint8_t* digest_unit, int j0, int nvalid, int lane,
                                           const uint32_t (&bmm)[16][2], const uint32_t (&bme)[8][2], float (&c)[4]) {
  const int g = lane >> 2, t = lane & 3;
  const int r0 = j0 + g, r1 = j0 + g + 8;
  const uint8_t* p0 = digest_unit + (int64_t)r0 * 512 + t * 16;
  const uint8_t* p1 = digest_unit + (int64_t)r1 * 512 + t * 16;
  uint4 v0[8], v1[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v0[i] = r0 < nvalid ? ldg_stream(p0 + i * 64) : make_uint4(0, 0, 0, 0);
    v1[i] = r1 < nvalid ? ldg_stream(p1 + i * 64) : make_uint4(0, 0, 0, 0);
  }
  c[0] = c[1] = c[2] = c[3] = 0.f;
  if (KIND == SCOUT_DIGEST_MINMAX) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      mma_bf16(c, v0[i].x, v1[i].x, v0[i].y, v1[i].y, bmm[2 * i][0], bmm[2 * i][1]);
      mma_bf16(c, v0[i].z, v1[i].z, v0[i].w, v1[i].w, bmm[2 * i + 1][0], bmm[2 * i + 1][1]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // four fp32 channels per row, each split exactly as hi + mid + lo (bf16)
      const float x0[4] = {__uint_as_float(v0[i].x), __uint_as_float(v0[i].y), __uint_as_float(v0[i].z),
                           __uint_as_float(v0[i].w)};
      const float x1[4] = {__uint_as_float(v1[i].x), __uint_as_float(v1[i].y), __uint_as_float(v1[i].z),
                           __uint_as_float(v1[i].w)};
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
        mma_bf16(c, A0, A1, A2, A3, bme[i][0], bme[i][1]);
      }
    }
  }
}

// Exclusive prefix over the CTA of four counters per thread; returns the totals.
__device__ __forceinline__ int4 block_excl_scan4(int4 v, int4* wsum, int4& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int4 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, inc.x, o), y = __shfl_up_sync(0xffffffffu, inc.y, o);
    const int z = __shfl_up_sync(0xffffffffu, inc.z, o), w = __shfl_up_sync(0xffffffffu, inc.w, o);
    if (lane >= o) {
      inc.x += x;
      inc.y += y;
      inc.z += z;
      inc.w += w;
    }
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int4 base = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
  for (int w = 0; w < kWarps; ++w) {
    const int4 s = wsum[w];
    if (w < warp) {
      base.x += s.x;
      base.y += s.y;
      base.z += s.z;
      base.w += s.w;
    }
    tot.x += s.x;
    tot.y += s.y;
    tot.z += s.z;
    tot.w += s.w;
  }
  __syncthreads();
  total = tot;
  return make_int4(base.x + inc.x - v.x, base.y + inc.y - v.y, base.z + inc.z - v.z, base.w + inc.w - v.w);
}

struct TopkArgs {
  const __nv_bfloat16* q;
  const uint8_t* digest;
  const int32_t* seq_len;
  const uint32_t* resident_bits;
  const int32_t* prev_list;
  const int32_t* prev_count;
  int Hq, Hkv, G, P, nblk_cap, k, words;
  float* scores;  // user buffer or workspace
  int32_t* counters;
  int32_t *topk_idx, *topk_count, *res_list, *res_count, *cpu_list, *cpu_count, *delta_list, *delta_count;
};

template <int KIND>
__global__ void __launch_bounds__(kThreads) score_topk_kernel(const TopkArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ __align__(16) __nv_bfloat16 qs[kMaxG * kD];
  __shared__ int4 wsum[kWarps];
  __shared__ int hist[256];
  __shared__ int s_last, s_digit, s_remaining;

  const int u = blockIdx.y;
  const int b = u / a.Hkv, kvh = u - b * a.Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvalid = min(a.nblk_cap, (max(a.seq_len[b], 0) + a.P - 1) / a.P);
  float* sc = a.scores + (int64_t)u * a.nblk_cap;

  // ---------------- phase 1: score this CTA's chunk ------------------------
  const int j0 = blockIdx.x * kChunk + warp * 16;
  const bool any = blockIdx.x * kChunk < nvalid;
  if (any) {
    const __nv_bfloat16* qg = a.q + ((int64_t)b * a.Hq + (int64_t)kvh * a.G) * kD;
    for (int i = threadIdx.x; i < a.G * kD; i += kThreads) qs[i] = qg[i];
  }
  __syncthreads();
  if (j0 < a.nblk_cap) {
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    if (j0 < nvalid) {
      uint32_t bmm[16][2], bme[8][2];
      const size_t row_bytes = 512;
      const uint8_t* du = a.digest + (int64_t)u * a.nblk_cap * row_bytes;
      if (KIND == SCOUT_DIGEST_MINMAX) {
        minmax_b_frag(qs, a.G, lane, bmm);
      } else {
        mean_b_frag(qs, a.G, lane, bme);
      }
      score_tile<KIND>(du, j0, nvalid, lane, bmm, bme, c);
    }
    // pool over the heads of the group (columns 2t, 2t+1 < G), then across t
    const int t = lane & 3, g = lane >> 2;
    const float ninf = -INFINITY;
    float m0 = fmaxf(2 * t < a.G ? c[0] : ninf, 2 * t + 1 < a.G ? c[1] : ninf);
    float m1 = fmaxf(2 * t < a.G ? c[2] : ninf, 2 * t + 1 < a.G ? c[3] : ninf);
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
    if (t == 0) {
      const int r0 = j0 + g, r1 = j0 + g + 8;
      if (r0 < a.nblk_cap) sc[r0] = r0 < nvalid ? m0 : ninf;
      if (r1 < a.nblk_cap) sc[r1] = r1 < nvalid ? m1 : ninf;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&a.counters[u], 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---------------- phase 2: select (last CTA of the unit) -----------------
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
  uint32_t* rbits = keys + a.nblk_cap;
  uint32_t* pbits = rbits + a.words;
  for (int j = threadIdx.x; j < nvalid; j += kThreads) keys[j] = score_key(__ldcg(sc + j));
  for (int w = threadIdx.x; w < a.words; w += kThreads) {
    rbits[w] = a.resident_bits[(int64_t)u * a.words + w];
    pbits[w] = 0u;
  }
  __syncthreads();
  if (a.prev_list != nullptr) {
    const int pc = min(max(a.prev_count[u], 0), a.k);
    for (int i = threadIdx.x; i < pc; i += kThreads) {
      const int j = a.prev_list[(int64_t)u * a.k + i];
      if (j >= 0 && j < a.nblk_cap) atomicOr(&pbits[j >> 5], 1u << (j & 31));
    }
  }
  const int keff = min(a.k, nvalid);
  uint32_t thr = 0u;  // every key of a finite score is > 0, so thr = 0 keeps all
  int need_eq = 0;
  if (keff < nvalid) {
    uint32_t prefix = 0u, mask = 0u;
    int remaining = keff;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += kThreads) hist[i] = 0;
      __syncthreads();
      for (int j = threadIdx.x; j < nvalid; j += kThreads) {
        const uint32_t key = keys[j];
        if (((key ^ prefix) & mask) == 0u) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns bins 255 - 8l .. 248 - 8l (high bins first)
        int cnt[8], sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          cnt[e] = hist[255 - 8 * lane - e];
          sum += cnt[e];
        }
        int inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += x;
        }
        const int before = inc - sum;  // keys in higher bins than this lane's
        if (before < remaining && remaining <= inc) {
          int acc = before;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (acc < remaining && remaining <= acc + cnt[e]) {
              s_digit = 255 - 8 * lane - e;
              s_remaining = remaining - acc;
            }
            acc += cnt[e];
          }
        }
      }
      __syncthreads();
      prefix |= (uint32_t)s_digit << shift;
      mask |= 255u << shift;
      remaining = s_remaining;
      __syncthreads();
    }
    thr = prefix;
    need_eq = remaining;
  }

  // ordered compaction: each thread owns a contiguous range of blocks, so the
  // lists come out in ascending block order
  const int per = (nvalid + kThreads - 1) / kThreads;
  const int lo = min(nvalid, (int)threadIdx.x * per), hi = min(nvalid, lo + per);
  int n_eq = 0;
  for (int j = lo; j < hi; ++j) n_eq += keys[j] == thr;
  int4 tot;
  const int eq_base = block_excl_scan4(make_int4(n_eq, 0, 0, 0), wsum, tot).x;
  int4 cnt = make_int4(0, 0, 0, 0);
  int eqr = eq_base;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = keys[j];
    const bool sel = key > thr || (key == thr && eqr < need_eq);
    eqr += key == thr;
    if (!sel) continue;
    const bool res = (rbits[j >> 5] >> (j & 31)) & 1u;
    cnt.x += 1;
    if (res) {
      cnt.y += 1;
    } else {
      cnt.z += 1;
      cnt.w += ((pbits[j >> 5] >> (j & 31)) & 1u) ? 0 : 1;
    }
  }
  int4 pos = block_excl_scan4(cnt, wsum, tot);
  const int64_t lb = (int64_t)u * a.k;
  eqr = eq_base;
  for (int j = lo; j < hi; ++j) {
    const uint32_t key = keys[j];
    const bool sel = key > thr || (key == thr && eqr < need_eq);
    eqr += key == thr;
    if (!sel) continue;
    a.topk_idx[lb + pos.x++] = j;
    if ((rbits[j >> 5] >> (j & 31)) & 1u) {
      a.res_list[lb + pos.y++] = j;
    } else {
      a.cpu_list[lb + pos.z++] = j;
      if (!((pbits[j >> 5] >> (j & 31)) & 1u)) a.delta_list[lb + pos.w++] = j;
    }
  }
  for (int i = threadIdx.x; i < a.k; i += kThreads) {
    if (i >= tot.x) a.topk_idx[lb + i] = -1;
    if (i >= tot.y) a.res_list[lb + i] = -1;
    if (i >= tot.z) a.cpu_list[lb + i] = -1;
    if (i >= tot.w) a.delta_list[lb + i] = -1;
  }
  if (threadIdx.x == 0) {
    a.topk_count[u] = tot.x;
    a.res_count[u] = tot.y;
    a.cpu_count[u] = tot.z;
    a.delta_count[u] = tot.w;
    a.counters[u] = 0;  // ready for the next call
  }
}

inline size_t counters_bytes(int64_t units) { return (size_t)((units * 4 + 255) / 256 * 256); }

}  // namespace
}  // namespace scout

extern "C" size_t scout_score_topk_workspace_bytes(int B, int Hkv, int nblk_cap) {
  if (B <= 0 || Hkv <= 0 || nblk_cap <= 0) return 0;
  const int64_t units = (int64_t)B * Hkv;
  return scout::counters_bytes(units) + (size_t)units * nblk_cap * sizeof(float);
}

extern "C" int scout_score_topk(int kind, const void* q, const void* digest, const int32_t* seq_len,
                                const uint32_t* resident_bits, const int32_t* prev_cpu_list,
                                const int32_t* prev_cpu_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap,
                                int k, float* scores, int32_t* topk_idx, int32_t* topk_count, int32_t* res_list,
                                int32_t* res_count, int32_t* cpu_list, int32_t* cpu_count, int32_t* delta_list,
                                int32_t* delta_count, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  using namespace scout;
  if (q == nullptr || digest == nullptr || seq_len == nullptr || resident_bits == nullptr || topk_idx == nullptr ||
      topk_count == nullptr || res_list == nullptr || res_count == nullptr || cpu_list == nullptr ||
      cpu_count == nullptr || delta_list == nullptr || delta_count == nullptr)
    return SCOUT_ERR_INVALID_ARG;
  if ((prev_cpu_list == nullptr) != (prev_cpu_count == nullptr)) return SCOUT_ERR_INVALID_ARG;
  if (kind != SCOUT_DIGEST_MINMAX && kind != SCOUT_DIGEST_MEAN) return SCOUT_ERR_INVALID_ARG;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || nblk_cap <= 0 || k <= 0) return SCOUT_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  const int64_t units = (int64_t)B * Hkv;
  if (D != kD || !valid_P(P) || G > kMaxG || nblk_cap > kMaxNblk || units > 65535 || !aligned16(digest))
    return SCOUT_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < scout_score_topk_workspace_bytes(B, Hkv, nblk_cap))
    return SCOUT_ERR_WORKSPACE;
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
  a.counters = static_cast<int32_t*>(workspace);
  a.scores = scores != nullptr ? scores
                               : reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + counters_bytes(units));
  a.topk_idx = topk_idx;
  a.topk_count = topk_count;
  a.res_list = res_list;
  a.res_count = res_count;
  a.cpu_list = cpu_list;
  a.cpu_count = cpu_count;
  a.delta_list = delta_list;
  a.delta_count = delta_count;
  const size_t smem = (size_t)(nblk_cap + 2 * a.words) * sizeof(uint32_t);
  const dim3 grid((unsigned)((nblk_cap + kChunk - 1) / kChunk), (unsigned)units);
  if (kind == SCOUT_DIGEST_MINMAX)
    score_topk_kernel<SCOUT_DIGEST_MINMAX><<<grid, kThreads, smem, stream>>>(a);
  else
    score_topk_kernel<SCOUT_DIGEST_MEAN><<<grid, kThreads, smem, stream>>>(a);
  return launch_status();
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
#include <mutex>

namespace scout {
namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB: counters + fp32 scores
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kNoAllocMaxDevices] = {};

// Device address of g_topk_scratch on the current device, looked up once per
// device (the host-side symbol is only a stand-in and must never reach a kernel).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SCOUT_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return SCOUT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || p == nullptr) return SCOUT_ERR_CUDA;
    g_scratch_addr[dev] = p;
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
                                        int32_t* delta_list, int32_t* delta_count, cudaStream_t stream) {
  using namespace scout;
  const size_t need = scout_score_topk_workspace_bytes(B, Hkv, nblk_cap);
  if (need == 0) return SCOUT_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return SCOUT_ERR_WORKSPACE;  // beyond the fixed scratch
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != SCOUT_OK) return rc;
  // the array keeps whatever the previous call left: zero the per-unit counters
  if (cudaMemsetAsync(scratch, 0, counters_bytes((int64_t)B * Hkv), stream) != cudaSuccess) return SCOUT_ERR_CUDA;
  return scout_score_topk(kind, q, digest, seq_len, resident_bits, prev_cpu_list, prev_cpu_count, B, Hq, Hkv, D, P,
                          nblk_cap, k, scores, topk_idx, topk_count, res_list, res_count, cpu_list, cpu_count,
                          delta_list, delta_count, scratch, kNoAllocScratchBytes, stream);
}
