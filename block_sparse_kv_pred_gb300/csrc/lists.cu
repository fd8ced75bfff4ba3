// scout_resident_list: every resident valid block of each unit, as a list the attention
// kernel can take.  ScoutAttention (arXiv HTML), Algorithm 1 (GPUATTN(Q, B_gpu)) read as
// "all blocks in GPU memory", the variant of the section 3.2 reading (the selected ones).
//
// One warp per unit: the lanes take 32 words (1024 blocks) at a time, count their set bits,
// and an exclusive scan over the lanes gives each lane its write position, so the list comes
// out ascending with coalesced reads of the bitmap.
#include "common.cuh"

namespace scout {
namespace {

__global__ void __launch_bounds__(256) resident_list_kernel(const uint32_t* __restrict__ bits,
                                                            const int32_t* __restrict__ seq_len, int units, int Hkv,
                                                            int P, int nblk_cap, int words, int cap,
                                                            int32_t* __restrict__ list, int32_t* __restrict__ count,
                                                            int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int u = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (u >= units) return;
  const int L = seq_len[u / Hkv];
  const int nvalid = min(nblk_cap, (max(L, 0) + P - 1) / P);
  const uint32_t* ub = bits + (int64_t)u * words;
  int32_t* ul = list + (int64_t)u * cap;
  int n = 0;  // entries found so far (the same on every lane)
  for (int w0 = 0; w0 * 32 < nvalid; w0 += 32) {
    const int w = w0 + lane;
    uint32_t m = 0u;
    if (w < words && w * 32 < nvalid) {
      m = ub[w];
      const int left = nvalid - w * 32;  // valid blocks in this word
      if (left < 32) m &= (1u << left) - 1u;
    }
    const int c = __popc(m);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    for (int pos = n + incl - c; m != 0u; m &= m - 1u, ++pos)
      if (pos < cap) ul[pos] = w * 32 + __ffs(m) - 1;
    n += __shfl_sync(0xffffffffu, incl, 31);
  }
  const int written = min(n, cap);
  for (int i = written + lane; i < cap; i += 32) ul[i] = -1;
  if (lane == 0) {
    count[u] = written;
    if (n > cap) report(status, SCOUT_DEV_OVERFLOW);
  }
}

}  // namespace
}  // namespace scout

extern "C" int scout_resident_list(const uint32_t* resident_bits, const int32_t* seq_len, int B, int Hkv, int P,
                                   int nblk_cap, int cap, int32_t* list, int32_t* count, int32_t* dev_status,
                                   cudaStream_t stream) {
  using namespace scout;
  if (resident_bits == nullptr || seq_len == nullptr || list == nullptr || count == nullptr || B <= 0 || Hkv <= 0 ||
      nblk_cap <= 0 || cap <= 0)
    return SCOUT_ERR_INVALID_ARG;
  if (!valid_P(P)) return SCOUT_ERR_UNSUPPORTED;
  const int64_t units = (int64_t)B * Hkv;
  if (units > 0x7fffffffLL / 32) return SCOUT_ERR_UNSUPPORTED;
  const int blocks = (int)((units + 7) / 8);
  resident_list_kernel<<<blocks, 256, 0, stream>>>(resident_bits, seq_len, (int)units, Hkv, P, nblk_cap,
                                                  (nblk_cap + 31) / 32, cap, list, count, dev_status);
  return launch_status();
}
