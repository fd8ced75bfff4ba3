// Asynchronous periodic recall (host side) and the residency commit.
// ScoutAttention (arXiv HTML), section 3.4: important blocks are copied back from
// host memory into GPU memory after a layer's attention, on a path that does not
// block inference; they are first needed at the same layer of the next step.
//
// Two ways to move the bytes, both on a side stream: plain cudaMemcpyAsync calls (one
// per run of consecutive blocks landing in consecutive slots; any pinned memory), or
// one gather kernel that reads the recalled pages straight from mapped pinned host
// memory (over NVLink-C2C on a Grace host) and writes them into their slots, so that
// scattered 8 KB pages do not pay a copy call each.  Page table and residency bits
// change only in scout_commit_residency, which the caller orders after the copies'
// event, so a block never looks resident before its bytes have landed.
#include <algorithm>
#include <cmath>
#include <utility>
#include <vector>

#include "common.cuh"

namespace scout {
namespace {

__global__ void commit_kernel(const scout_recall_op* __restrict__ ops, int n, int32_t* __restrict__ page_table,
                              uint32_t* __restrict__ bits, int64_t n_slots, int units, int nblk_cap, int words) {
  // a single CTA: evictions first, then insertions, so a slot handed over
  // within one recall ends up owned by its new block
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const scout_recall_op op = ops[i];
    if (op.unit < 0 || op.unit >= units || op.evict_block < 0 || op.evict_block >= nblk_cap) continue;
    page_table[(int64_t)op.unit * nblk_cap + op.evict_block] = -1;
    atomicAnd(&bits[(int64_t)op.unit * words + (op.evict_block >> 5)], ~(1u << (op.evict_block & 31)));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const scout_recall_op op = ops[i];
    if (op.unit < 0 || op.unit >= units || op.block < 0 || op.block >= nblk_cap || op.slot < 0 || op.slot >= n_slots)
      continue;
    page_table[(int64_t)op.unit * nblk_cap + op.block] = op.slot;
    atomicOr(&bits[(int64_t)op.unit * words + (op.block >> 5)], 1u << (op.block & 31));
  }
}

// One warp per (op, K or V page): the page's 16-byte chunks, four loads in flight per lane
// before the stores, from the host copy [units][nblk_cap][P][D] into the pool slot.
// An op outside the tables or the pool is skipped and reported.
__global__ void __launch_bounds__(256) recall_gather_kernel(const scout_recall_op* __restrict__ ops, int n,
                                                            const uint4* __restrict__ hK, const uint4* __restrict__ hV,
                                                            uint4* __restrict__ K_pool, uint4* __restrict__ V_pool,
                                                            int64_t n_slots, int units, int nblk_cap, int chunks,
                                                            int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < 2 * (int64_t)n; w += warps) {
    const scout_recall_op op = ops[w >> 1];
    if (op.unit < 0 || op.unit >= units || op.block < 0 || op.block >= nblk_cap || op.slot < 0 ||
        op.slot >= n_slots) {
      if (lane == 0 && (w & 1) == 0) report(status, SCOUT_DEV_BAD_INDEX);
      continue;
    }
    const uint4* src = ((w & 1) ? hV : hK) + ((int64_t)op.unit * nblk_cap + op.block) * chunks;
    uint4* dst = ((w & 1) ? V_pool : K_pool) + (int64_t)op.slot * chunks;
    for (int c = lane; c < chunks; c += 128) {
      uint4 v[4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (c + 32 * r < chunks) v[r] = ldg_stream(src + c + 32 * r);
#pragma unroll
      for (int r = 0; r < 4; ++r)
        if (c + 32 * r < chunks) dst[c + 32 * r] = v[r];
    }
  }
}

// Device address of a host range [p, p + bytes) in pinned, mapped host memory, or nullptr.
void* mapped_address(const void* p, size_t bytes) {
  cudaPointerAttributes first, last;
  const uint8_t* end = static_cast<const uint8_t*>(p) + bytes - 1;
  if (cudaPointerGetAttributes(&first, p) != cudaSuccess || cudaPointerGetAttributes(&last, end) != cudaSuccess) {
    cudaGetLastError();  // the lookup's error is this call's answer, not a sticky launch error
    return nullptr;
  }
  if (first.type != cudaMemoryTypeHost || last.type != cudaMemoryTypeHost || first.devicePointer == nullptr ||
      last.devicePointer == nullptr ||
      static_cast<const uint8_t*>(last.devicePointer) - static_cast<const uint8_t*>(first.devicePointer) !=
          static_cast<ptrdiff_t>(bytes - 1))
    return nullptr;
  return first.devicePointer;
}

int check_recall(int n_ops, const void* ops, const void* host_K, const void* host_V, const void* K_pool,
                 const void* V_pool, int64_t n_slots, int B, int Hkv, int D, int P, int nblk_cap,
                 const scout_launch* launch) {
  if (n_ops < 0 || (n_ops > 0 && ops == nullptr) || host_K == nullptr || host_V == nullptr || K_pool == nullptr ||
      V_pool == nullptr || B <= 0 || Hkv <= 0 || nblk_cap <= 0 || n_slots <= 0)
    return SCOUT_ERR_INVALID_ARG;
  if (launch != nullptr && (launch->inject != SCOUT_INJECT_NONE && launch->inject != SCOUT_INJECT_COPY_FAIL))
    return SCOUT_ERR_INVALID_ARG;
  if (D != kD || !valid_P(P)) return SCOUT_ERR_UNSUPPORTED;
  return SCOUT_OK;
}

}  // namespace
}  // namespace scout

extern "C" int scout_recall_async(const scout_recall_op* ops, int n_ops, const void* host_K, const void* host_V,
                                  void* K_pool, void* V_pool, int64_t n_slots, int B, int Hkv, int D, int P,
                                  int nblk_cap, const scout_launch* launch, cudaEvent_t wait_event,
                                  cudaStream_t side_stream, cudaEvent_t done_event) {
  using namespace scout;
  const int rc = check_recall(n_ops, ops, host_K, host_V, K_pool, V_pool, n_slots, B, Hkv, D, P, nblk_cap, launch);
  if (rc != SCOUT_OK) return rc;
  const bool fail_copy = launch != nullptr && launch->inject == SCOUT_INJECT_COPY_FAIL;
  const int64_t units = (int64_t)B * Hkv;
  for (int i = 0; i < n_ops; ++i) {
    const scout_recall_op& op = ops[i];
    if (op.unit < 0 || op.unit >= units || op.block < 0 || op.block >= nblk_cap || op.slot < 0 || op.slot >= n_slots ||
        op.evict_block < -1 || op.evict_block >= nblk_cap)
      return SCOUT_ERR_INVALID_ARG;
  }
  if (wait_event != nullptr && cudaStreamWaitEvent(side_stream, wait_event, 0) != cudaSuccess) return SCOUT_ERR_CUDA;
  const size_t page = (size_t)P * kD * 2;
  const auto* hK = static_cast<const uint8_t*>(host_K);
  const auto* hV = static_cast<const uint8_t*>(host_V);
  auto* dK = static_cast<uint8_t*>(K_pool);
  auto* dV = static_cast<uint8_t*>(V_pool);
  int i = 0, runs = 0;
  while (i < n_ops) {
    // extend the run while source blocks and destination slots are both consecutive
    int r = 1;
    while (i + r < n_ops && ops[i + r].unit == ops[i].unit && ops[i + r].block == ops[i].block + r &&
           ops[i + r].slot == ops[i].slot + r)
      ++r;
    const size_t src = ((size_t)ops[i].unit * nblk_cap + ops[i].block) * page;
    const size_t dst = (size_t)ops[i].slot * page;
    if (fail_copy && runs++ == 1) return SCOUT_ERR_CUDA;  // as if this run's copy had been refused
    if (cudaMemcpyAsync(dK + dst, hK + src, page * r, cudaMemcpyHostToDevice, side_stream) != cudaSuccess ||
        cudaMemcpyAsync(dV + dst, hV + src, page * r, cudaMemcpyHostToDevice, side_stream) != cudaSuccess)
      return SCOUT_ERR_CUDA;
    i += r;
  }
  if (done_event != nullptr && cudaEventRecord(done_event, side_stream) != cudaSuccess) return SCOUT_ERR_CUDA;
  return SCOUT_OK;
}

extern "C" int scout_recall_gather_async(const scout_recall_op* d_ops, int n_ops, const void* host_K,
                                         const void* host_V, void* K_pool, void* V_pool, int64_t n_slots, int B,
                                         int Hkv, int D, int P, int nblk_cap, int32_t* dev_status,
                                         const scout_launch* launch, cudaEvent_t wait_event, cudaStream_t side_stream,
                                         cudaEvent_t done_event) {
  using namespace scout;
  const int rc = check_recall(n_ops, d_ops, host_K, host_V, K_pool, V_pool, n_slots, B, Hkv, D, P, nblk_cap, launch);
  if (rc != SCOUT_OK) return rc;
  if (!aligned16(host_K) || !aligned16(host_V) || !aligned16(K_pool) || !aligned16(V_pool))
    return SCOUT_ERR_UNSUPPORTED;
  // the device addresses of the host copies: both ends of each must lie in pinned host memory
  // mapped into the device's address space (cudaHostAlloc / cudaMallocHost, or cudaHostRegister
  // on a unified-addressing system), at the same offset from one another on the device
  const size_t bytes = (size_t)B * Hkv * nblk_cap * P * kD * 2;
  void* dK = mapped_address(host_K, bytes);
  void* dV = mapped_address(host_V, bytes);
  if (dK == nullptr || dV == nullptr) return SCOUT_ERR_UNSUPPORTED;
  if (launch != nullptr && launch->inject == SCOUT_INJECT_COPY_FAIL) return SCOUT_ERR_CUDA;  // as if refused
  if (wait_event != nullptr && cudaStreamWaitEvent(side_stream, wait_event, 0) != cudaSuccess) return SCOUT_ERR_CUDA;
  if (n_ops > 0) {
    const int chunks = P * kD * 2 / 16;
    const int64_t warps_needed = 2 * (int64_t)n_ops;
    const int grid = (int)std::min<int64_t>((warps_needed + 7) / 8, (int64_t)sm_count() * 8);
    recall_gather_kernel<<<grid, 256, 0, side_stream>>>(d_ops, n_ops, static_cast<const uint4*>(dK),
                                                       static_cast<const uint4*>(dV), static_cast<uint4*>(K_pool),
                                                       static_cast<uint4*>(V_pool), n_slots, B * Hkv, nblk_cap,
                                                       chunks, dev_status);
    if (launch_status() != SCOUT_OK) return SCOUT_ERR_CUDA;
  }
  if (done_event != nullptr && cudaEventRecord(done_event, side_stream) != cudaSuccess) return SCOUT_ERR_CUDA;
  return SCOUT_OK;
}

extern "C" int scout_commit_residency(const scout_recall_op* d_ops, int n_ops, int32_t* page_table,
                                      uint32_t* resident_bits, int64_t n_slots, int B, int Hkv, int nblk_cap,
                                      cudaEvent_t wait_event, cudaStream_t stream) {
  using namespace scout;
  if (n_ops < 0 || (n_ops > 0 && d_ops == nullptr) || page_table == nullptr || resident_bits == nullptr || B <= 0 ||
      Hkv <= 0 || nblk_cap <= 0 || n_slots <= 0)
    return SCOUT_ERR_INVALID_ARG;
  if (wait_event != nullptr && cudaStreamWaitEvent(stream, wait_event, 0) != cudaSuccess) return SCOUT_ERR_CUDA;
  if (n_ops == 0) return SCOUT_OK;
  commit_kernel<<<1, 1024, 0, stream>>>(d_ops, n_ops, page_table, resident_bits, n_slots, B * Hkv, nblk_cap,
                                        (nblk_cap + 31) / 32);
  return launch_status();
}

// Host-side plan of one recall step.  Per unit: the selected blocks that are not
// resident come in, the most important first (score descending, lower block first);
// each takes the slot of a resident block that is not selected, the least important
// first (score ascending, lower block first); the unit's resident set keeps its size.
extern "C" int scout_plan_recall(const float* scores, const int32_t* topk_idx, const int32_t* topk_count,
                                 const uint32_t* resident_bits, const int32_t* page_table, int units, int nblk_cap,
                                 int k, scout_recall_op* ops, int max_ops, int* n_ops) {
  if (scores == nullptr || topk_idx == nullptr || topk_count == nullptr || resident_bits == nullptr ||
      page_table == nullptr || n_ops == nullptr || units <= 0 || nblk_cap <= 0 || k <= 0 || max_ops < 0 ||
      (ops == nullptr && max_ops > 0))
    return SCOUT_ERR_INVALID_ARG;
  const int words = (nblk_cap + 31) / 32;
  std::vector<char> sel(nblk_cap);
  std::vector<int> in, ev;
  int n = 0;
  for (int u = 0; u < units; ++u) {
    const float* U = scores + (int64_t)u * nblk_cap;
    const uint32_t* bits = resident_bits + (int64_t)u * words;
    auto resident = [&](int j) { return ((bits[j >> 5] >> (j & 31)) & 1u) != 0; };
    std::fill(sel.begin(), sel.end(), 0);
    const int cnt = std::min(std::max(topk_count[u], 0), k);
    for (int i = 0; i < cnt; ++i) {
      const int j = topk_idx[(int64_t)u * k + i];
      if (j < 0 || j >= nblk_cap) return SCOUT_ERR_INVALID_ARG;
      sel[j] = 1;
    }
    in.clear();
    ev.clear();
    for (int j = 0; j < nblk_cap; ++j) {
      if (sel[j] && !resident(j)) in.push_back(j);
      if (!sel[j] && resident(j)) ev.push_back(j);
    }
    // exact comparisons of the fp32 scores; equal scores fall back to the block index
    std::stable_sort(in.begin(), in.end(), [&](int x, int y) { return U[x] > U[y]; });
    std::stable_sort(ev.begin(), ev.end(), [&](int x, int y) { return U[x] < U[y]; });
    const size_t m = std::min(in.size(), ev.size());
    const int first = n;
    for (size_t i = 0; i < m; ++i) {
      const int32_t slot = page_table[(int64_t)u * nblk_cap + ev[i]];
      if (slot < 0) return SCOUT_ERR_INVALID_ARG;  // a resident block must own a slot
      if (n >= max_ops) return SCOUT_ERR_WORKSPACE;
      ops[n++] = scout_recall_op{u, in[i], slot, ev[i]};
    }
    std::sort(ops + first, ops + n, [](const scout_recall_op& x, const scout_recall_op& y) { return x.block < y.block; });
  }
  *n_ops = n;
  return SCOUT_OK;
}

// Recall plan with residency per page (one block of a sequence for all its KV heads): the
// pages some head selects that are not resident come in, the most important first (the largest
// of the heads' scores); each takes the slots of a resident page no head selects, the least
// important first; one op per KV head and pair.
extern "C" int scout_plan_recall_pages(const float* scores, const int32_t* topk_idx, const int32_t* topk_count,
                                       const uint32_t* resident_bits, const int32_t* page_table, int B, int Hkv,
                                       int nblk_cap, int k, scout_recall_op* ops, int max_ops, int* n_ops) {
  if (scores == nullptr || topk_idx == nullptr || topk_count == nullptr || resident_bits == nullptr ||
      page_table == nullptr || n_ops == nullptr || B <= 0 || Hkv <= 0 || nblk_cap <= 0 || k <= 0 || max_ops < 0 ||
      (ops == nullptr && max_ops > 0))
    return SCOUT_ERR_INVALID_ARG;
  const int words = (nblk_cap + 31) / 32;
  std::vector<char> sel(nblk_cap);
  std::vector<float> imp(nblk_cap);
  std::vector<int> in, ev;
  std::vector<std::pair<int, int>> pairs;
  int n = 0;
  for (int b = 0; b < B; ++b) {
    const int u0 = b * Hkv;
    const uint32_t* bits = resident_bits + (int64_t)u0 * words;
    for (int h = 1; h < Hkv; ++h)  // one residency per page: every head's bits are the same
      if (!std::equal(bits, bits + words, resident_bits + (int64_t)(u0 + h) * words)) return SCOUT_ERR_INVALID_ARG;
    auto resident = [&](int j) { return ((bits[j >> 5] >> (j & 31)) & 1u) != 0; };
    std::fill(sel.begin(), sel.end(), 0);
    for (int j = 0; j < nblk_cap; ++j) {
      float m = scores[(int64_t)u0 * nblk_cap + j];
      for (int h = 1; h < Hkv; ++h) m = std::max(m, scores[(int64_t)(u0 + h) * nblk_cap + j]);
      imp[j] = m;
    }
    for (int h = 0; h < Hkv; ++h) {
      const int u = u0 + h;
      const int cnt = std::min(std::max(topk_count[u], 0), k);
      for (int i = 0; i < cnt; ++i) {
        const int j = topk_idx[(int64_t)u * k + i];
        if (j < 0 || j >= nblk_cap) return SCOUT_ERR_INVALID_ARG;
        sel[j] = 1;
      }
    }
    in.clear();
    ev.clear();
    for (int j = 0; j < nblk_cap; ++j) {
      if (sel[j] && !resident(j)) in.push_back(j);
      if (!sel[j] && resident(j)) ev.push_back(j);
    }
    std::stable_sort(in.begin(), in.end(), [&](int x, int y) { return imp[x] > imp[y]; });
    std::stable_sort(ev.begin(), ev.end(), [&](int x, int y) { return imp[x] < imp[y]; });
    pairs.clear();
    for (size_t i = 0; i < std::min(in.size(), ev.size()); ++i) pairs.emplace_back(in[i], ev[i]);
    std::sort(pairs.begin(), pairs.end());  // ascending incoming block
    for (int h = 0; h < Hkv; ++h) {
      const int u = u0 + h;
      for (const auto& pr : pairs) {
        const int32_t slot = page_table[(int64_t)u * nblk_cap + pr.second];
        if (slot < 0) return SCOUT_ERR_INVALID_ARG;  // a resident page owns a slot in every head
        if (n >= max_ops) return SCOUT_ERR_WORKSPACE;
        ops[n++] = scout_recall_op{u, pr.first, slot, pr.second};
      }
    }
  }
  *n_ops = n;
  return SCOUT_OK;
}

// Per-layer recall intervals (section 3.4): for each layer, the number of leading profiled
// steps whose CPU compute ratio stays below beta, at least 1 and at most the profile's length.
extern "C" int scout_recall_intervals(const float* ratio, int layers, int steps, float beta, int32_t* interval) {
  if (ratio == nullptr || interval == nullptr || layers <= 0 || steps <= 0 || !(beta > 0.f) || !std::isfinite(beta))
    return SCOUT_ERR_INVALID_ARG;
  for (int l = 0; l < layers; ++l) {
    const float* r = ratio + (int64_t)l * steps;
    int n = 0;
    while (n < steps && r[n] < beta) ++n;  // a NaN is not below beta
    interval[l] = n > 0 ? n : 1;
  }
  return SCOUT_OK;
}
