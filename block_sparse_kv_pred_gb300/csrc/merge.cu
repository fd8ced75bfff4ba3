// scout_merge: LSE-weighted combination of the GPU and CPU partial results.
// ScoutAttention (arXiv HTML), section 3.2: the two devices' intermediate results
// are merged on the GPU with the FlashAttention (online-softmax) rule.
//
// One warp per query-head row, 4 channels per lane (float4), fully coalesced.
#include "common.cuh"

namespace scout {
namespace {

constexpr int kRowsPerCta = 8;

__global__ void __launch_bounds__(kRowsPerCta * 32) merge_kernel(const float* __restrict__ Oa, const float* __restrict__ La,
                                                                 const float* __restrict__ Ob, const float* __restrict__ Lb,
                                                                 int rows, __nv_bfloat16* __restrict__ Out,
                                                                 float* __restrict__ Lout) {
  const int row = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float la = La[row], lb = Lb[row];
  const float m = fmaxf(la, lb);
  float wa = 0.f, wb = 0.f, lse = -INFINITY;
  if (m != -INFINITY) {
    wa = expf(la - m);
    wb = expf(lb - m);
    const float s = wa + wb;
    lse = m + logf(s);
    wa /= s;
    wb /= s;
  }
  const float4 a = reinterpret_cast<const float4*>(Oa + (int64_t)row * kD)[lane];
  const float4 b = reinterpret_cast<const float4*>(Ob + (int64_t)row * kD)[lane];
  uint2 o;
  o.x = pack_bf16(wa * a.x + wb * b.x, wa * a.y + wb * b.y);
  o.y = pack_bf16(wa * a.z + wb * b.z, wa * a.w + wb * b.w);
  reinterpret_cast<uint2*>(Out + (int64_t)row * kD)[lane] = o;
  if (Lout != nullptr && lane == 0) Lout[row] = lse;
}

}  // namespace
}  // namespace scout

extern "C" int scout_merge(const float* O_a, const float* lse_a, const float* O_b, const float* lse_b, int rows, int D,
                           void* O_out, float* lse_out, cudaStream_t stream) {
  using namespace scout;
  if (O_a == nullptr || lse_a == nullptr || O_b == nullptr || lse_b == nullptr || O_out == nullptr)
    return SCOUT_ERR_INVALID_ARG;
  if (rows < 0) return SCOUT_ERR_INVALID_ARG;
  if (D != kD || !aligned16(O_a) || !aligned16(O_b) || (reinterpret_cast<uintptr_t>(O_out) & 7u))
    return SCOUT_ERR_UNSUPPORTED;
  if (rows == 0) return SCOUT_OK;
  merge_kernel<<<(rows + kRowsPerCta - 1) / kRowsPerCta, kRowsPerCta * 32, 0, stream>>>(
      O_a, lse_a, O_b, lse_b, rows, static_cast<__nv_bfloat16*>(O_out), lse_out);
  return launch_status();
}
