// scout_predict_q: layer-ahead query prediction Q_pred = X W_Q^T.
// ScoutAttention (arXiv HTML), section 3.3 and Algorithm 1 (query prediction):
// the next layer's query projection applied to the current layer's input.
//
// Shared-memory tiled GEMM on the CUDA cores: a CTA computes a 32 x 32 tile of
// Q (rows of X x rows of W), fp32 accumulation, bf16 output.
#include "common.cuh"

namespace scout {
namespace {

constexpr int kTile = 32, kKt = 64;

__global__ void __launch_bounds__(256) predict_q_simple(const __nv_bfloat16* __restrict__ X,
                                                        const __nv_bfloat16* __restrict__ W,
                                                        __nv_bfloat16* __restrict__ Q, int M, int N, int K) {
  __shared__ float xs[kTile][kKt + 1], ws[kTile][kKt + 1];
  const int n0 = blockIdx.x * kTile, m0 = blockIdx.y * kTile;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // ty: 0..7
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = 0; k0 < K; k0 += kKt) {
    for (int e = threadIdx.x; e < kTile * kKt; e += 256) {
      const int r = e / kKt, c = e - r * kKt;
      xs[r][c] = (m0 + r < M && k0 + c < K) ? __bfloat162float(X[(int64_t)(m0 + r) * K + k0 + c]) : 0.f;
      ws[r][c] = (n0 + r < N && k0 + c < K) ? __bfloat162float(W[(int64_t)(n0 + r) * K + k0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < kKt; ++c) {
      const float w = ws[tx][c];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = fmaf(xs[ty + 8 * i][c], w, acc[i]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 8 * i, n = n0 + tx;
    if (m < M && n < N) Q[(int64_t)m * N + n] = __float2bfloat16_rn(acc[i]);
  }
}

}  // namespace
}  // namespace scout

extern "C" int scout_predict_q(const void* X, const void* W, void* Q, int M, int N, int K, cudaStream_t stream) {
  using namespace scout;
  if (X == nullptr || W == nullptr || Q == nullptr || M <= 0 || N <= 0 || K <= 0) return SCOUT_ERR_INVALID_ARG;
  if (M > 256 || N % 128 != 0 || K % 64 != 0 || !aligned16(X) || !aligned16(W) || !aligned16(Q))
    return SCOUT_ERR_UNSUPPORTED;
  const dim3 grid((unsigned)(N / kTile), (unsigned)((M + kTile - 1) / kTile));
  predict_q_simple<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(X),
                                             static_cast<const __nv_bfloat16*>(W), static_cast<__nv_bfloat16*>(Q), M,
                                             N, K);
  return launch_status();
}
