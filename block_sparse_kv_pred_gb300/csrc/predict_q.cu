// scout_predict_q: layer-ahead query prediction Q_pred = X W_Q^T on the 5th-generation
// tensor cores.  ScoutAttention (arXiv HTML), section 3.3 and Algorithm 1 (query
// prediction): the next layer's query projection applied to the current layer's input.
//
// Decode batches are small (M = 1..256 rows of X) while W_Q is large, so the GEMM is
// computed swapped: D[n][m] = sum_k W[n][k] X[m][k].  A CTA owns 128 rows of W (the
// MMA's M = 128 TMEM lanes); the batch, padded to a multiple of 16, is the MMA's N.
// W and X tiles (64 k-columns, 128-byte swizzle) stream in by TMA through a ring of
// shared-memory stages guarded by mbarriers, up to four k-blocks per stage (measured on
// GB300: one k-block per stage streams ~25% slower, the barrier round trip of a stage
// being paid per 22 KB instead of per 88 KB); one thread issues tcgen05.mma into a
// TMEM accumulator and frees each stage with tcgen05.commit.  The K dimension is
// split over the CTAs of a thread-block cluster so that about one CTA runs per SM.
// The batch columns of the accumulator are dealt out over the cluster's CTAs: each
// CTA stores the columns another CTA owns straight into that CTA's shared memory
// (distributed shared memory), then sums the partials of its own columns and writes
// them as bf16 Q.  No global scratch is used.

#include "common.cuh"

namespace scout {
namespace {

constexpr int kBM = 128;      // W rows per CTA (MMA M)
constexpr int kBK = 64;       // k columns per k-block (one 128-byte swizzle atom of bf16)
constexpr int kMaxKps = 4;    // k-blocks per ring stage, at most
constexpr int kStages = 16;  // upper bound; the ring takes what shared memory holds
constexpr int kThreadsQ = 128;
constexpr int kMaxN = 256;    // padded batch (MMA N) limit
constexpr int kWTileBytes = kBM * kBK * 2;  // 16 KiB

// --- cluster PTX --------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_peer(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Instruction descriptor: fp32 accumulate, bf16 A and B, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

struct GemmArgs {
  __nv_bfloat16* Q;
  int M, N, n_pad, tmem_cols, kblocks, stages, x_tile_bytes;
  int kps;  // k-blocks per ring stage
  int32_t* status;
};

// A ring stage holds nk <= kps consecutive k-blocks: their W tiles first, then their X tiles.
// One arrival expects both; the W and the X copies may be issued apart.
__device__ __forceinline__ void load_w(uint8_t* st, const CUtensorMap* tmW, const GemmArgs& a, int tile, int kb,
                                       int nk, uint64_t* bar) {
  mbar_arrive_tx(bar, (uint32_t)(nk * (kWTileBytes + a.x_tile_bytes)));
  for (int j = 0; j < nk; ++j) tma_load_2d(st + j * kWTileBytes, tmW, (kb + j) * kBK, tile * kBM, bar);
}
__device__ __forceinline__ void load_x(uint8_t* st, const CUtensorMap* tmX, const GemmArgs& a, int kb, int nk,
                                       uint64_t* bar) {
  for (int j = 0; j < nk; ++j)
    tma_load_2d(st + a.kps * kWTileBytes + j * a.x_tile_bytes, tmX, (kb + j) * kBK, 0, bar);
}

__global__ void __launch_bounds__(kThreadsQ, 1) predict_q_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                 const __grid_constant__ CUtensorMap tmX,
                                                                 const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full_bar[kStages], empty_bar[kStages], done_bar;
  __shared__ uint32_t tmem_slot;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int stage_bytes = a.kps * (kWTileBytes + a.x_tile_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;
  const uint32_t S = gridDim.y, rank = cluster_rank();
  const int kb0 = (int)(rank * a.kblocks / S), kb1 = (int)((rank + 1) * a.kblocks / S);
  const int nst = (kb1 - kb0 + a.kps - 1) / a.kps;  // ring stages of this CTA's k range
  auto nk_of = [&](int i) { return min(a.kps, kb1 - kb0 - i * a.kps); };
  // a kernel that starts early after this one (scout_score_topk) may take SMs as they free up;
  // it waits for this grid to finish before it reads Q
  release_dependents();

  // the first pass over the ring needs no free slot: issue it before the TMEM allocation.  W
  // does not depend on an earlier kernel; X may be written by the one this launch follows, so
  // an early start waits for it between the two
  const int first = min(a.stages, nst);
  if (tid == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(&done_bar, 1);
    fence_mbar_init();
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
    for (int i = 0; i < first; ++i)
      load_w(base + i * stage_bytes, &tmW, a, tile, kb0 + i * a.kps, nk_of(i), &full_bar[i]);
    wait_prerequisites();
    for (int i = 0; i < first; ++i) load_x(base + i * stage_bytes, &tmX, a, kb0 + i * a.kps, nk_of(i), &full_bar[i]);
  }
  if (warp == 2) tmem_alloc(&tmem_slot, (uint32_t)a.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0 && lane == 0) {
    // TMA producer: the rest of the k range, each stage once the MMAs have freed it
    int issued = first;
    for (int i = first; i < nst; ++i) {
      const int st = i % a.stages;
      if (!mbar_wait(&empty_bar[st], ((i / a.stages) & 1) ^ 1)) {
        report(a.status, SCOUT_DEV_TIMEOUT);
        break;
      }
      load_w(base + st * stage_bytes, &tmW, a, tile, kb0 + i * a.kps, nk_of(i), &full_bar[st]);
      load_x(base + st * stage_bytes, &tmX, a, kb0 + i * a.kps, nk_of(i), &full_bar[st]);
      issued = i + 1;
    }
    // every issued copy lands before the CTA can retire
    for (int r = 0; r < a.stages && r < issued; ++r) {
      const int last = issued - 1 - r;
      if (!mbar_wait(&full_bar[last % a.stages], (last / a.stages) & 1)) report(a.status, SCOUT_DEV_TIMEOUT);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    const uint32_t idesc = idesc_bf16(a.n_pad);
    for (int i = 0; i < nst; ++i) {
      const int st = i % a.stages;
      if (!mbar_wait(&full_bar[st], (i / a.stages) & 1)) {
        report(a.status, SCOUT_DEV_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t s0 = smem_u32(base + st * stage_bytes);
      const int nk = nk_of(i);
      for (int j = 0; j < nk; ++j) {
        const uint32_t sW = s0 + j * kWTileBytes, sX = s0 + a.kps * kWTileBytes + j * a.x_tile_bytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          umma_bf16(tmem, sw128_desc(sW + kk * 32), sw128_desc(sX + kk * 32), idesc,
                    (i > 0 || j > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&empty_bar[st]);
    }
    umma_commit(&done_bar);
  }
  __syncwarp();

  // ---- epilogue: thread (warp w, lane l) owns W row tile*128 + 32w + l (TMEM lane) ----
  // Column group g (8 batch columns) belongs to CTA g % S of the cluster.  recv holds, for
  // every source CTA s and every group this CTA owns, s's partial: [S][owned][8][128] fp32.
  if (!mbar_wait(&done_bar, 0)) report(a.status, SCOUT_DEV_TIMEOUT);
  tc_fence_after();
  const int r_local = warp * 32 + lane;
  const int row = tile * kBM + r_local;
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
  const int ngroups = a.n_pad / 8;
  const int owned = (ngroups + (int)S - 1) / (int)S;
  float* recv = reinterpret_cast<float*>(base);  // the stage ring is idle now
  float v[8];
  if (S > 1) {
    cluster_sync();  // every CTA of the cluster is done with its ring: it may be written
    for (int g = 0; g < ngroups; ++g) {
      const uint32_t owner = (uint32_t)g % S;
      if (owner == rank) continue;
      tmem_ld8(trow + (uint32_t)(g * 8), v);
      const int slot = ((int)rank * owned + g / (int)S) * 8;
      const uint32_t dst = map_peer(smem_u32(recv + slot * kBM + r_local), owner);
#pragma unroll
      for (int e = 0; e < 8; ++e) st_peer(dst + (uint32_t)(e * kBM * 4), v[e]);
    }
    cluster_sync();  // the partials have landed (release/acquire across the cluster)
  }
  for (int g = (int)rank; g < ngroups; g += (int)S) {
    tmem_ld8(trow + (uint32_t)(g * 8), v);
    for (uint32_t s = 0; s < S; ++s) {
      if (s == rank) continue;
      const float* src = recv + ((int)s * owned + g / (int)S) * 8 * kBM + r_local;
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] += src[e * kBM];
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int m = g * 8 + e;
      if (m < a.M && row < a.N) a.Q[(int64_t)m * a.N + row] = __float2bfloat16_rn(v[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
}

bool make_map(CUtensorMap* map, const void* ptr, int rows, int cols, int box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace scout

extern "C" int scout_predict_q(const void* X, const void* W, void* Q, int M, int N, int K, int32_t* dev_status,
                               const scout_launch* launch, cudaStream_t stream) {
  using namespace scout;
  if (X == nullptr || W == nullptr || Q == nullptr || M <= 0 || N <= 0 || K <= 0) return SCOUT_ERR_INVALID_ARG;
  if (launch != nullptr && launch->max_ctas < 0) return SCOUT_ERR_INVALID_ARG;
  if (M > kMaxN || N % kBM != 0 || K % kBK != 0 || !aligned16(X) || !aligned16(W) || !aligned16(Q))
    return SCOUT_ERR_UNSUPPORTED;
  GemmArgs a;
  a.Q = static_cast<__nv_bfloat16*>(Q);
  a.M = M;
  a.N = N;
  a.n_pad = (M + 15) / 16 * 16;
  a.tmem_cols = 32;
  while (a.tmem_cols < a.n_pad) a.tmem_cols <<= 1;
  a.kblocks = K / kBK;
  a.x_tile_bytes = (a.n_pad * 128 + 1023) / 1024 * 1024;
  // ~220 KB in flight per SM, in stages of up to kMaxKps k-blocks (the fewer the stages, the
  // fewer barrier round trips per byte) but at least two, so that copies and MMAs overlap
  constexpr int kRingBytes = 224 * 1024;
  a.kps = max(1, min(kMaxKps, kRingBytes / 2 / (kWTileBytes + a.x_tile_bytes)));
  const int stage_bytes = a.kps * (kWTileBytes + a.x_tile_bytes);
  a.stages = min(kStages, kRingBytes / stage_bytes);
  a.status = dev_status;
  const int tiles = N / kBM;
  const int cap = launch != nullptr && launch->max_ctas > 0 ? launch->max_ctas : sm_count();
  const int S = max(1, min(min(8, a.kblocks), cap / tiles));  // split-K so tiles x S fits the CTA budget
  const int owned = (a.n_pad / 8 + S - 1) / S;                  // column groups per CTA in the reduction
  const size_t smem = 1024 + (size_t)max(a.stages * stage_bytes, S * owned * 8 * kBM * 4);
  CUtensorMap tmW, tmX;
  if (!make_map(&tmW, W, N, K, kBM) || !make_map(&tmX, X, M, K, a.n_pad)) return SCOUT_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(predict_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return SCOUT_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles, (unsigned)S, 1);
  cfg.blockDim = dim3(kThreadsQ, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)S;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early_start_attrs(launch, attr, 1);
  if (cudaLaunchKernelEx(&cfg, predict_q_kernel, tmW, tmX, a) != cudaSuccess) return SCOUT_ERR_CUDA;
  return launch_status();
}
