// Asynchronous periodic recall (host side) and the residency commit.
// ScoutAttention (arXiv HTML), section 3.4: important blocks are copied back from
// host memory into GPU memory after a layer's attention, on a path that does not
// block inference; they are first needed at the same layer of the next step.
//
// The copies run on a side stream as plain cudaMemcpyAsync calls (one per run of
// consecutive blocks landing in consecutive slots).  Page table and residency
// bits change only in scout_commit_residency, which the caller orders after the
// copies' event, so a block never looks resident before its bytes have landed.
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

}  // namespace
}  // namespace scout

extern "C" int scout_recall_async(const scout_recall_op* ops, int n_ops, const void* host_K, const void* host_V,
                                  void* K_pool, void* V_pool, int64_t n_slots, int B, int Hkv, int D, int P,
                                  int nblk_cap, cudaEvent_t wait_event, cudaStream_t side_stream,
                                  cudaEvent_t done_event) {
  using namespace scout;
  if (n_ops < 0 || (n_ops > 0 && ops == nullptr) || host_K == nullptr || host_V == nullptr || K_pool == nullptr ||
      V_pool == nullptr || B <= 0 || Hkv <= 0 || nblk_cap <= 0 || n_slots <= 0)
    return SCOUT_ERR_INVALID_ARG;
  if (D != kD || !valid_P(P)) return SCOUT_ERR_UNSUPPORTED;
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
  int i = 0;
  while (i < n_ops) {
    // extend the run while source blocks and destination slots are both consecutive
    int r = 1;
    while (i + r < n_ops && ops[i + r].unit == ops[i].unit && ops[i + r].block == ops[i].block + r &&
           ops[i + r].slot == ops[i].slot + r)
      ++r;
    const size_t src = ((size_t)ops[i].unit * nblk_cap + ops[i].block) * page;
    const size_t dst = (size_t)ops[i].slot * page;
    if (cudaMemcpyAsync(dK + dst, hK + src, page * r, cudaMemcpyHostToDevice, side_stream) != cudaSuccess ||
        cudaMemcpyAsync(dV + dst, hV + src, page * r, cudaMemcpyHostToDevice, side_stream) != cudaSuccess)
      return SCOUT_ERR_CUDA;
    i += r;
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
