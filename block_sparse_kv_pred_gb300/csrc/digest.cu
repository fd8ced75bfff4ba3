// scout_build_digest: per-block key digests over a paged bf16 KV cache.
// ScoutAttention (arXiv HTML), section 2.2: Quest min/max pooling, MoBA mean pooling.
//
// One warp per (unit, block).  Lane l reads 16 bytes (8 channels, chunk l % 16)
// of rows t = l / 16, l / 16 + 2, ...; the two half-warps are combined with a
// shuffle, so every K byte of the block is read exactly once, coalesced.
#include "common.cuh"

namespace scout {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void two_sum_add(float& s, float& c, float x) {
  // Neumaier's compensated summation step
  float t = s + x;
  if (fabsf(s) >= fabsf(x))
    c += (s - t) + x;
  else
    c += (x - t) + s;
  s = t;
}

template <int P, int KIND>
__global__ void __launch_bounds__(kWarps * 32) digest_kernel(const __nv_bfloat16* __restrict__ K_pool, int64_t n_slots,
                                                             const int32_t* __restrict__ page_table,
                                                             const int32_t* __restrict__ seq_len, int Hkv,
                                                             int64_t units, int nblk_cap, int64_t n_items,
                                                             const int32_t* __restrict__ block_list, void* digest,
                                                             int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (item >= n_items) return;
  int64_t u, j;
  if (block_list != nullptr) {
    u = block_list[2 * item];
    j = block_list[2 * item + 1];
  } else {
    u = item / nblk_cap;
    j = item - u * nblk_cap;
  }
  if (u < 0 || j < 0 || j >= nblk_cap || u >= units) {
    if (lane == 0) report(status, SCOUT_DEV_BAD_INDEX);
    return;
  }
  const int b = (int)(u / Hkv);
  const int len = seq_len[b];
  const int valid = min(P, len - (int)(j * P));
  if (valid <= 0) return;  // block holds no tokens: left untouched
  const int32_t slot = page_table[u * nblk_cap + j];
  if (slot < 0 || slot >= n_slots) {
    if (lane == 0) report(status, SCOUT_DEV_BAD_INDEX);
    return;
  }
  const int half = lane >> 4, chunk = lane & 15;
  const __nv_bfloat16* base = K_pool + ((int64_t)slot * P) * kD + chunk * 8;

  float a[8], c[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    a[e] = KIND == SCOUT_DIGEST_MINMAX ? __int_as_float(0x7f800000) : 0.f;  // min (or sum)
    c[e] = KIND == SCOUT_DIGEST_MINMAX ? __int_as_float(0xff800000) : 0.f;  // max (or compensation)
  }
  constexpr int kRows = P / 2;
  constexpr int kBatch = kRows < 8 ? kRows : 8;
#pragma unroll
  for (int r0 = 0; r0 < kRows; r0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int t = 2 * (r0 + i) + half;
      v[i] = t < valid ? ldg_stream(base + (int64_t)t * kD) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int t = 2 * (r0 + i) + half;
      if (t >= valid) continue;
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float x = (e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]);
        if (KIND == SCOUT_DIGEST_MINMAX) {
          a[e] = fminf(a[e], x);
          c[e] = fmaxf(c[e], x);
        } else {
          two_sum_add(a[e], c[e], x);
        }
      }
    }
  }
  // combine the two half-warps (rows of even and odd parity)
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float pa = __shfl_xor_sync(0xffffffffu, a[e], 16);
    const float pc = __shfl_xor_sync(0xffffffffu, c[e], 16);
    if (KIND == SCOUT_DIGEST_MINMAX) {
      a[e] = fminf(a[e], pa);
      c[e] = fmaxf(c[e], pc);
    } else {
      float s = a[e], comp = c[e] + pc;
      two_sum_add(s, comp, pa);
      a[e] = (s + comp) / (float)valid;
    }
  }
  const int64_t blk = u * nblk_cap + j;
  if (KIND == SCOUT_DIGEST_MINMAX) {
    // lanes 0-15 write the min row, lanes 16-31 the max row: one 512-byte store
    const float* src = half ? c : a;
    uint4 o;
    o.x = pack_bf16(src[0], src[1]);
    o.y = pack_bf16(src[2], src[3]);
    o.z = pack_bf16(src[4], src[5]);
    o.w = pack_bf16(src[6], src[7]);
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(digest) + blk * 2 * kD + half * kD + chunk * 8)[0] = o;
  } else if (half == 0) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(digest) + blk * kD + chunk * 8);
    dst[0] = make_float4(a[0], a[1], a[2], a[3]);
    dst[1] = make_float4(a[4], a[5], a[6], a[7]);
  }
}

template <int P>
int launch_digest(int kind, const void* K_pool, int64_t n_slots, const int32_t* page_table, const int32_t* seq_len,
                  int Hkv, int64_t units, int nblk_cap, int64_t n_items, const int32_t* block_list, void* digest, int32_t* status,
                  cudaStream_t st) {
  const dim3 grid((unsigned)((n_items + kWarps - 1) / kWarps));
  auto Kp = static_cast<const __nv_bfloat16*>(K_pool);
  if (kind == SCOUT_DIGEST_MINMAX)
    digest_kernel<P, SCOUT_DIGEST_MINMAX><<<grid, kWarps * 32, 0, st>>>(Kp, n_slots, page_table, seq_len, Hkv,
                                                                      units, nblk_cap, n_items, block_list, digest, status);
  else
    digest_kernel<P, SCOUT_DIGEST_MEAN><<<grid, kWarps * 32, 0, st>>>(Kp, n_slots, page_table, seq_len, Hkv,
                                                                    units, nblk_cap, n_items, block_list, digest, status);
  return launch_status();
}

}  // namespace
}  // namespace scout

extern "C" int scout_build_digest(int kind, const void* K_pool, int64_t n_slots, const int32_t* page_table,
                                  const int32_t* seq_len, int B, int Hkv, int D, int P, int nblk_cap,
                                  const int32_t* block_list, int n_list, void* digest, int32_t* dev_status,
                                  cudaStream_t stream) {
  using namespace scout;
  if (K_pool == nullptr || page_table == nullptr || seq_len == nullptr || digest == nullptr) return SCOUT_ERR_INVALID_ARG;
  if (B <= 0 || Hkv <= 0 || nblk_cap <= 0 || n_slots <= 0 || n_list < 0) return SCOUT_ERR_INVALID_ARG;
  if (kind != SCOUT_DIGEST_MINMAX && kind != SCOUT_DIGEST_MEAN) return SCOUT_ERR_INVALID_ARG;
  if (D != kD || !valid_P(P) || !aligned16(K_pool) || !aligned16(digest)) return SCOUT_ERR_UNSUPPORTED;
  const int64_t n_items = block_list != nullptr ? (int64_t)n_list : (int64_t)B * Hkv * nblk_cap;
  if (n_items == 0) return SCOUT_OK;
  switch (P) {
    case 16: return launch_digest<16>(kind, K_pool, n_slots, page_table, seq_len, Hkv, (int64_t)B * Hkv, nblk_cap, n_items, block_list, digest, dev_status, stream);
    case 32: return launch_digest<32>(kind, K_pool, n_slots, page_table, seq_len, Hkv, (int64_t)B * Hkv, nblk_cap, n_items, block_list, digest, dev_status, stream);
    default: return launch_digest<64>(kind, K_pool, n_slots, page_table, seq_len, Hkv, (int64_t)B * Hkv, nblk_cap, n_items, block_list, digest, dev_status, stream);
  }
}
