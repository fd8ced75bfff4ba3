// Device twin of the seeded input generator in workload/__init__.py.
//
// Only inputs are made here: the same SplitMix64 counter hash and Irwin-Hall(12)
// construction as the host generator, so a device-filled tensor equals the host
// one bit for bit.  This library is separate from libscout and holds none of the
// method's arithmetic.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float irwin_hall(uint64_t key, uint64_t idx) {
  uint64_t base = key + 3ull * idx;
  int total = 0;
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    uint64_t h = mix64(base + (uint64_t)r);
    total += (int)(h & 0xFFFF) + (int)((h >> 16) & 0xFFFF) + (int)((h >> 32) & 0xFFFF) + (int)(h >> 48);
  }
  // total < 2^20, so every step below is exact in fp32
  return __fsub_rn(__fmul_rn((float)total, 1.0f / 65536.0f), 6.0f);
}

__global__ void fill_normal_bf16(__nv_bfloat16* __restrict__ dst, int64_t n, uint64_t key, float sigma,
                                 int64_t offset) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    float z = irwin_hall(key, (uint64_t)(offset + i));
    dst[i] = __float2bfloat16_rn(__fmul_rn(z, sigma));
  }
}

// pool[slot][p][d]: slot s holds block j of unit u where owner[s] = u * nblk + j.
__global__ void fill_pool_bf16(__nv_bfloat16* __restrict__ pool, int64_t n_slots, int P, int D,
                               const int32_t* __restrict__ owner, int nblk, uint64_t key,
                               const float* __restrict__ chan_scale, const uint8_t* __restrict__ heavy,
                               const float* __restrict__ hdir) {
  const int64_t per_slot = (int64_t)P * D;
  const int64_t n = n_slots * per_slot;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    int64_t s = e / per_slot;
    int64_t r = e - s * per_slot;
    int p = (int)(r / D), d = (int)(r - (int64_t)p * D);
    int32_t own = owner[s];
    int64_t u = own / nblk, j = own - u * nblk;
    int64_t t = j * P + p;
    uint64_t idx = (uint64_t)((u * nblk * P + t) * D + d);
    float x = __fmul_rn(irwin_hall(key, idx), chan_scale[d]);
    if (heavy != nullptr && heavy[u * nblk + j]) x = __fadd_rn(x, hdir[u * D + d]);
    pool[e] = __float2bfloat16_rn(x);
  }
}

uint64_t host_mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t key_of(uint64_t seed, uint64_t stream) { return host_mix64(host_mix64(seed) ^ stream); }

int grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  if (g > 152 * 64) g = 152 * 64;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

#define GEN_API __attribute__((visibility("default")))

extern "C" {

// Fill dst[0..n) with bf16(z * sigma), z the Irwin-Hall variate of counter offset + i.
GEN_API int scoutgen_fill_normal_bf16(void* dst, int64_t n, uint64_t seed, uint64_t stream, float sigma, int64_t offset,
                              cudaStream_t st) {
  if (n <= 0) return 0;
  fill_normal_bf16<<<grid_for(n), 256, 0, st>>>((__nv_bfloat16*)dst, n, key_of(seed, stream), sigma, offset);
  return (int)cudaGetLastError();
}

// Fill a paged K or V pool from the logical per-unit tensors (see Workload.unit_kv).
GEN_API int scoutgen_fill_pool_bf16(void* pool, int64_t n_slots, int P, int D, const int32_t* owner, int nblk, uint64_t seed,
                            uint64_t stream, const float* chan_scale, const uint8_t* heavy, const float* hdir,
                            cudaStream_t st) {
  if (n_slots <= 0) return 0;
  fill_pool_bf16<<<grid_for(n_slots * P * D), 256, 0, st>>>((__nv_bfloat16*)pool, n_slots, P, D, owner, nblk,
                                                          key_of(seed, stream), chan_scale, heavy, hdir);
  return (int)cudaGetLastError();
}

}  // extern "C"
