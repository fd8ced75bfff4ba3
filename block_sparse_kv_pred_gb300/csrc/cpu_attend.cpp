// scout_cpu_attend: attention over the offloaded blocks on the host cores.
// ScoutAttention (arXiv HTML), section 3.2 and Algorithm 1 (CPUAttn of B_cpu, spawned one
// layer ahead): the selected blocks that are not resident on the GPU are attended on the CPU,
// next to the host copy of the KV cache, with the predicted query; the GPU merges the result.
//
// The threads take whole units (sequence, KV head) from an atomic counter, the units with the
// longest CPU lists first (so that the threads finish together).  For a unit, the G
// query rows are held in fp32, and a block-wise online softmax rescales the running sums to
// each block's maximum.  Two implementations of a unit:
//
// * the tiled one (the default), written with the compiler's generic 4 x fp32 vectors (GCC
//   vector extensions: NEON on AArch64, SSE on x86-64; no intrinsics, no target flags):
//   bf16 widened by interleaving with zero halves (a zip per four values), scores in register
//   tiles of TT tokens x G heads (G q rows against TT widened K rows, 8 dimensions per step,
//   one horizontal sum per score at the end), then the block's V accumulated in register
//   tiles of 16 (8 for more than six heads) dimensions x G heads over every token of the
//   block, the running sums loaded, rescaled and stored once per tile (tiles sized for
//   AArch64's 32 vector registers).  Measured on the Grace cores against the first version
//   of this form, which widened bf16 by a vector conversion: 7.2 against 4.0 GB/s on one core
//   (the conversion compiled to lane-by-lane inserts); an exponential of its own, four
//   weights at a time, and a software prefetch of the next block did not help;
// * the scalar one (scout_cpu_attend_scalar), plain loops with 16 partial sums per product,
//   the reference the tiled one is tested against.
#if !defined(__GNUC__)
#error "the tiled CPU attention uses GCC/Clang vector extensions"
#endif
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <thread>
#include <vector>

#include "scout.h"

namespace {

constexpr int kDim = 128;      // head dimension
constexpr int kMaxGroup = 8;   // query heads per KV head
constexpr int kMaxPage = 64;   // tokens per block
constexpr int kLanes = 16;     // partial sums per dot product

inline float fold(float (&p)[kLanes]) {  // sum of the partial sums, pairwise
  for (int w = kLanes / 2; w > 0; w /= 2)
    for (int e = 0; e < w; ++e) p[e] += p[e + w];
  return p[0];
}

inline float widen(uint16_t v) {  // bf16 -> fp32 (exact)
  const uint32_t u = static_cast<uint32_t>(v) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return f;
}

struct Job {
  const uint16_t* q;
  const uint16_t* K;
  const uint16_t* V;
  const int32_t* seq_len;
  const int32_t* list;
  const int32_t* count;
  int Hq, Hkv, G, P, nblk_cap, k;
  float scale;
  float* O;
  float* lse;
};

typedef float f32x4 __attribute__((vector_size(16)));
typedef uint16_t u16x8 __attribute__((vector_size(16)));

// Eight bf16 -> two vectors of four fp32 (exact): a bf16 is the upper half of its fp32, so each
// value is interleaved with a zero half (a zip with a zero vector; one instruction per half on
// AArch64).  The element order of the vector types is the memory order on both targets.
inline void widen8(const uint16_t* p, f32x4& lo, f32x4& hi) {
  u16x8 h;
  std::memcpy(&h, p, sizeof h);
  const u16x8 z = {0, 0, 0, 0, 0, 0, 0, 0};
  const u16x8 a = __builtin_shuffle(z, h, (u16x8){0, 8, 1, 9, 2, 10, 3, 11});
  const u16x8 c = __builtin_shuffle(z, h, (u16x8){4, 12, 5, 13, 6, 14, 7, 15});
  std::memcpy(&lo, &a, sizeof lo);
  std::memcpy(&hi, &c, sizeof hi);
}

inline float hsum(f32x4 v) { return (v[0] + v[1]) + (v[2] + v[3]); }

// One unit with register tiles; G query heads per KV head (a template argument, so that the
// tiles are fixed-size arrays the compiler keeps in registers).
template <int G>
void attend_unit_tiled(const Job& a, int u) {
  constexpr int TT = G <= 4 ? 4 : (G <= 6 ? 3 : 2);  // tokens per score tile: G x TT accumulators
  constexpr int DV = G <= 6 ? 4 : 2;                  // 4-wide vectors per V tile: G x DV accumulators
  const int b = u / a.Hkv, kvh = u - b * a.Hkv, P = a.P;
  alignas(64) f32x4 q[G][kDim / 4];
  alignas(64) f32x4 acc[G][kDim / 4];
  alignas(64) float s[G][kMaxPage + 4];
  float m[G], l[G], corr[G];
  const uint16_t* qg = a.q + (static_cast<int64_t>(b) * a.Hq + static_cast<int64_t>(kvh) * G) * kDim;
  for (int h = 0; h < G; ++h) {
    for (int c = 0; c < kDim / 4; c += 2) {
      widen8(qg + h * kDim + 4 * c, q[h][c], q[h][c + 1]);
      acc[h][c] = acc[h][c + 1] = f32x4{0.f, 0.f, 0.f, 0.f};
    }
    m[h] = -INFINITY;
    l[h] = 0.f;
  }
  const int L = a.seq_len[b];
  const int n = a.count[u];
  const int32_t* blocks = a.list + static_cast<int64_t>(u) * a.k;
  for (int i = 0; i < n; ++i) {
    const int j = blocks[i];
    const int valid = std::min(P, L - j * P);
    if (valid <= 0) continue;  // no token of this block is in the sequence yet
    const int64_t base = (static_cast<int64_t>(u) * a.nblk_cap + j) * P * kDim;
    const uint16_t* Kb = a.K + base;
    const uint16_t* Vb = a.V + base;
    // scores: tiles of TT tokens (rows past the valid ones stay inside the block's P rows; their
    // scores are computed and never used)
    for (int t0 = 0; t0 < valid; t0 += TT) {
      f32x4 c[G][TT];
      for (int h = 0; h < G; ++h)
        for (int x = 0; x < TT; ++x) c[h][x] = f32x4{0.f, 0.f, 0.f, 0.f};
      // TT need not divide P: the last tile of a block re-reads its last rows (in bounds; the
      // scores of rows past P are never used)
      const int r0 = std::min(t0, P - TT);
      for (int d = 0; d < kDim / 4; d += 2) {
        f32x4 k0[TT], k1[TT];
        for (int x = 0; x < TT; ++x) widen8(Kb + (r0 + x) * kDim + 4 * d, k0[x], k1[x]);
        for (int h = 0; h < G; ++h)
          for (int x = 0; x < TT; ++x) c[h][x] += q[h][d] * k0[x];
        for (int h = 0; h < G; ++h)
          for (int x = 0; x < TT; ++x) c[h][x] += q[h][d + 1] * k1[x];
      }
      for (int h = 0; h < G; ++h)
        for (int x = 0; x < TT; ++x) s[h][r0 + x] = a.scale * hsum(c[h][x]);
    }
    // online softmax: s becomes the probabilities, corr the factor of the running sums
    for (int h = 0; h < G; ++h) {
      float mb = m[h];
      for (int x = 0; x < valid; ++x) mb = std::max(mb, s[h][x]);
      corr[h] = m[h] == -INFINITY ? 0.f : std::exp(m[h] - mb);
      float sum = 0.f;
      for (int x = 0; x < valid; ++x) {
        s[h][x] = std::exp(s[h][x] - mb);
        sum += s[h][x];
      }
      l[h] = l[h] * corr[h] + sum;
      m[h] = mb;
    }
    // acc_h = corr_h acc_h + sum_t p_h(t) v_t, one tile of 4 * DV dimensions at a time
    for (int c0 = 0; c0 < kDim / 4; c0 += DV) {
      f32x4 r[G][DV];
      for (int h = 0; h < G; ++h)
        for (int e = 0; e < DV; ++e) r[h][e] = acc[h][c0 + e] * corr[h];
      for (int t = 0; t < valid; ++t) {
        f32x4 v[DV];
        for (int e = 0; e < DV; e += 2) widen8(Vb + t * kDim + 4 * (c0 + e), v[e], v[e + 1]);
        for (int h = 0; h < G; ++h) {
          const float w = s[h][t];
          for (int e = 0; e < DV; ++e) r[h][e] += w * v[e];
        }
      }
      for (int h = 0; h < G; ++h)
        for (int e = 0; e < DV; ++e) acc[h][c0 + e] = r[h][e];
    }
  }
  for (int h = 0; h < G; ++h) {
    const int64_t row = static_cast<int64_t>(b) * a.Hq + static_cast<int64_t>(kvh) * G + h;
    const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
    for (int c = 0; c < kDim / 4; ++c) {
      const f32x4 o = acc[h][c] * inv;
      std::memcpy(a.O + row * kDim + 4 * c, &o, sizeof o);
    }
    a.lse[row] = l[h] > 0.f ? m[h] + std::log(l[h]) : -INFINITY;
  }
}

void attend_unit_scalar(const Job& a, int u);

// The implementation a job runs, by its group size.
using UnitFn = void (*)(const Job&, int);
UnitFn unit_fn(int G, bool scalar) {
  if (scalar) return attend_unit_scalar;
  switch (G) {
    case 1: return attend_unit_tiled<1>;
    case 2: return attend_unit_tiled<2>;
    case 3: return attend_unit_tiled<3>;
    case 4: return attend_unit_tiled<4>;
    case 5: return attend_unit_tiled<5>;
    case 6: return attend_unit_tiled<6>;
    case 7: return attend_unit_tiled<7>;
    default: return attend_unit_tiled<8>;
  }
}

void attend_unit_scalar(const Job& a, int u) {
  const int b = u / a.Hkv, kvh = u - b * a.Hkv, G = a.G, P = a.P;
  alignas(64) float q[kMaxGroup][kDim];
  alignas(64) float acc[kMaxGroup][kDim];
  alignas(64) float s[kMaxGroup][kMaxPage];
  alignas(64) float row[kDim];
  alignas(64) float vr[4][kDim];
  float m[kMaxGroup], l[kMaxGroup];
  const uint16_t* qg = a.q + (static_cast<int64_t>(b) * a.Hq + static_cast<int64_t>(kvh) * G) * kDim;
  for (int h = 0; h < G; ++h) {
    for (int d = 0; d < kDim; ++d) {
      q[h][d] = widen(qg[h * kDim + d]);
      acc[h][d] = 0.f;
    }
    m[h] = -INFINITY;
    l[h] = 0.f;
  }
  const int L = a.seq_len[b];
  const int n = a.count[u];
  const int32_t* blocks = a.list + static_cast<int64_t>(u) * a.k;
  for (int i = 0; i < n; ++i) {
    const int j = blocks[i];
    const int valid = std::min(P, L - j * P);
    if (valid <= 0) continue;  // no token of this block is in the sequence yet
    const int64_t base = (static_cast<int64_t>(u) * a.nblk_cap + j) * P * kDim;
    const uint16_t* Kb = a.K + base;
    const uint16_t* Vb = a.V + base;
    // scores s = scale * q_h . k_t
    int t = 0;
    for (; t < valid; ++t) {
      for (int d = 0; d < kDim; ++d) row[d] = widen(Kb[t * kDim + d]);
      for (int h = 0; h < G; ++h) {
        float p0[kLanes] = {};
        for (int d = 0; d < kDim; d += kLanes)
          for (int e = 0; e < kLanes; ++e) p0[e] += q[h][d + e] * row[d + e];
        s[h][t] = a.scale * fold(p0);
      }
    }
    // online softmax: the running sums move to the new maximum, s becomes the probabilities
    for (int h = 0; h < G; ++h) {
      float mb = m[h];
      for (int x = 0; x < valid; ++x) mb = std::max(mb, s[h][x]);
      const float corr = m[h] == -INFINITY ? 0.f : std::exp(m[h] - mb);
      float sum = 0.f;
      for (int x = 0; x < valid; ++x) {
        s[h][x] = std::exp(s[h][x] - mb);
        sum += s[h][x];
      }
      l[h] = l[h] * corr + sum;
      if (corr != 1.f)
        for (int d = 0; d < kDim; ++d) acc[h][d] *= corr;
      m[h] = mb;
    }
    // acc_h += p_h(t) v_t, four tokens per pass over acc_h
    for (t = 0; t + 4 <= valid; t += 4) {
      for (int d = 0; d < kDim; ++d) {
        vr[0][d] = widen(Vb[t * kDim + d]);
        vr[1][d] = widen(Vb[(t + 1) * kDim + d]);
        vr[2][d] = widen(Vb[(t + 2) * kDim + d]);
        vr[3][d] = widen(Vb[(t + 3) * kDim + d]);
      }
      for (int h = 0; h < G; ++h) {
        const float w0 = s[h][t], w1 = s[h][t + 1], w2 = s[h][t + 2], w3 = s[h][t + 3];
        for (int d = 0; d < kDim; ++d)
          acc[h][d] += (w0 * vr[0][d] + w1 * vr[1][d]) + (w2 * vr[2][d] + w3 * vr[3][d]);
      }
    }
    for (; t < valid; ++t) {
      for (int d = 0; d < kDim; ++d) row[d] = widen(Vb[t * kDim + d]);
      for (int h = 0; h < G; ++h) {
        const float w0 = s[h][t];
        for (int d = 0; d < kDim; ++d) acc[h][d] += w0 * row[d];
      }
    }
  }
  for (int h = 0; h < G; ++h) {
    const int64_t r = static_cast<int64_t>(b) * a.Hq + static_cast<int64_t>(kvh) * G + h;
    const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
    for (int d = 0; d < kDim; ++d) a.O[r * kDim + d] = acc[h][d] * inv;
    a.lse[r] = l[h] > 0.f ? m[h] + std::log(l[h]) : -INFINITY;
  }
}

// Every argument check of scout_cpu_attend; fills the job when they pass.
int make_job(const void* q, const void* K, const void* V, const int32_t* seq_len, const int32_t* cpu_list,
             const int32_t* cpu_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap, int k, float scale,
             float* O_cpu, float* lse_cpu, Job* job) {
  if (q == nullptr || K == nullptr || V == nullptr || seq_len == nullptr || cpu_list == nullptr ||
      cpu_count == nullptr || O_cpu == nullptr || lse_cpu == nullptr || B <= 0 || Hq <= 0 || Hkv <= 0 ||
      nblk_cap <= 0 || k <= 0 || Hq % Hkv != 0 || Hq / Hkv > kMaxGroup || !(scale > 0.f) || !std::isfinite(scale))
    return SCOUT_ERR_INVALID_ARG;
  if (D != kDim || (P != 16 && P != 32 && P != 64)) return SCOUT_ERR_UNSUPPORTED;
  const int units = B * Hkv;
  for (int u = 0; u < units; ++u) {  // every list is checked before anything is written
    const int n = cpu_count[u];
    if (n < 0 || n > k) return SCOUT_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
      const int j = cpu_list[static_cast<int64_t>(u) * k + i];
      if (j < 0 || j >= nblk_cap) return SCOUT_ERR_INVALID_ARG;
    }
  }
  *job = Job{static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(K), static_cast<const uint16_t*>(V),
             seq_len, cpu_list, cpu_count, Hq, Hkv, Hq / Hkv, P, nblk_cap, k, scale, O_cpu, lse_cpu};
  return SCOUT_OK;
}

// The order in which the threads take the units: the longest CPU lists first (ties by unit
// index), so that the last units dealt are short ones and the threads finish together.  The
// result of a unit does not depend on the thread that computes it.
void longest_first(const Job& a, int units, std::vector<int>& order) {
  order.resize(units);
  for (int u = 0; u < units; ++u) order[u] = u;
  std::stable_sort(order.begin(), order.end(), [&a](int x, int y) { return a.count[x] > a.count[y]; });
}

// scout_cpu_attend and scout_cpu_attend_scalar: threads started and joined by the call.
int attend_sync(const void* q, const void* K, const void* V, const int32_t* seq_len, const int32_t* cpu_list,
                const int32_t* cpu_count, int B, int Hq, int Hkv, int D, int P, int nblk_cap, int k, float scale,
                float* O_cpu, float* lse_cpu, int n_threads, bool scalar) {
  Job a;
  const int rc = make_job(q, K, V, seq_len, cpu_list, cpu_count, B, Hq, Hkv, D, P, nblk_cap, k, scale, O_cpu,
                          lse_cpu, &a);
  if (rc != SCOUT_OK) return rc;
  const int units = B * Hkv;
  int nt = n_threads > 0 ? n_threads : static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  nt = std::min(nt, units);
  std::vector<int> order;
  try {
    longest_first(a, units, order);
  } catch (...) {
    return SCOUT_ERR_INVALID_ARG;  // no memory for the order of B * Hkv units
  }
  std::atomic<int> next{0};
  const UnitFn fn = unit_fn(a.G, scalar);
  auto work = [&a, &next, &order, units, fn]() {
    for (int i = next.fetch_add(1); i < units; i = next.fetch_add(1)) fn(a, order[i]);
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < nt; ++i) {
    try {
      pool.emplace_back(work);
    } catch (...) {  // no thread to be had: the ones running (at least this one) do the rest
      break;
    }
  }
  work();
  for (auto& th : pool) th.join();
  return SCOUT_OK;
}

}  // namespace

extern "C" int scout_cpu_attend(const void* q, const void* K, const void* V, const int32_t* seq_len,
                                const int32_t* cpu_list, const int32_t* cpu_count, int B, int Hq, int Hkv, int D,
                                int P, int nblk_cap, int k, float scale, float* O_cpu, float* lse_cpu,
                                int n_threads) {
  return attend_sync(q, K, V, seq_len, cpu_list, cpu_count, B, Hq, Hkv, D, P, nblk_cap, k, scale, O_cpu, lse_cpu,
                     n_threads, false);
}

extern "C" int scout_cpu_attend_scalar(const void* q, const void* K, const void* V, const int32_t* seq_len,
                                       const int32_t* cpu_list, const int32_t* cpu_count, int B, int Hq, int Hkv,
                                       int D, int P, int nblk_cap, int k, float scale, float* O_cpu, float* lse_cpu,
                                       int n_threads) {
  return attend_sync(q, K, V, seq_len, cpu_list, cpu_count, B, Hq, Hkv, D, P, nblk_cap, k, scale, O_cpu, lse_cpu,
                     n_threads, true);
}

// ---------------------------------------------------------------------------
// A caller-owned pool of worker threads for the CPU side, so that a pipeline calling it every
// layer does not start and join threads each time, and can wait for a layer's partial with a
// bound (a late CPU partial is reported, not waited for without end).  One job at a time.
// ---------------------------------------------------------------------------
struct scout_cpu_pool {
  std::vector<std::thread> threads;
  std::mutex mu;
  std::condition_variable cv_work, cv_done;
  Job job{};
  int units = 0;
  std::vector<int> order;  // the current job's units, longest CPU list first
  std::atomic<int> next{0};
  unsigned generation = 0;  // bumped by every submission
  int active = 0;           // workers still on the current job
  bool running = false, stop = false;

  void worker() {
    unsigned seen = 0;
    for (;;) {
      Job j;
      int n;
      const int* ord;
      {
        std::unique_lock<std::mutex> lk(mu);
        cv_work.wait(lk, [&] { return stop || generation != seen; });
        if (stop) return;
        seen = generation;
        j = job;
        n = units;
        ord = order.data();  // not resized while the job runs
      }
      const UnitFn fn = unit_fn(j.G, false);
      for (int i = next.fetch_add(1); i < n; i = next.fetch_add(1)) fn(j, ord[i]);
      std::lock_guard<std::mutex> lk(mu);
      if (--active == 0) {
        running = false;
        cv_done.notify_all();
      }
    }
  }
};

extern "C" scout_cpu_pool* scout_cpu_pool_create(int n_threads) {
  const int nt = n_threads > 0 ? n_threads : static_cast<int>(std::max(1u, std::thread::hardware_concurrency()));
  scout_cpu_pool* p = nullptr;
  try {
    p = new scout_cpu_pool;
    for (int i = 0; i < nt; ++i) p->threads.emplace_back([p] { p->worker(); });
  } catch (...) {
    if (p != nullptr) scout_cpu_pool_destroy(p);
    return nullptr;
  }
  return p;
}

extern "C" int scout_cpu_pool_threads(const scout_cpu_pool* pool) {
  return pool == nullptr ? 0 : static_cast<int>(pool->threads.size());
}

extern "C" void scout_cpu_pool_destroy(scout_cpu_pool* pool) {
  if (pool == nullptr) return;
  {
    std::unique_lock<std::mutex> lk(pool->mu);
    pool->cv_done.wait(lk, [&] { return !pool->running; });  // a job in flight finishes first
    pool->stop = true;
  }
  pool->cv_work.notify_all();
  for (auto& th : pool->threads) th.join();
  delete pool;
}

extern "C" int scout_cpu_attend_async(scout_cpu_pool* pool, const void* q, const void* K, const void* V,
                                      const int32_t* seq_len, const int32_t* cpu_list, const int32_t* cpu_count,
                                      int B, int Hq, int Hkv, int D, int P, int nblk_cap, int k, float scale,
                                      float* O_cpu, float* lse_cpu) {
  if (pool == nullptr || pool->threads.empty()) return SCOUT_ERR_INVALID_ARG;
  Job a;
  const int rc = make_job(q, K, V, seq_len, cpu_list, cpu_count, B, Hq, Hkv, D, P, nblk_cap, k, scale, O_cpu,
                          lse_cpu, &a);
  if (rc != SCOUT_OK) return rc;
  {
    std::lock_guard<std::mutex> lk(pool->mu);
    if (pool->running) return SCOUT_ERR_INVALID_ARG;  // one job at a time: wait for the last one first
    try {
      longest_first(a, B * Hkv, pool->order);
    } catch (...) {
      return SCOUT_ERR_INVALID_ARG;  // no memory for the order of B * Hkv units
    }
    pool->job = a;
    pool->units = B * Hkv;
    pool->next.store(0);
    pool->active = static_cast<int>(pool->threads.size());
    pool->running = true;
    ++pool->generation;
  }
  pool->cv_work.notify_all();
  return SCOUT_OK;
}

extern "C" int scout_cpu_pool_wait(scout_cpu_pool* pool, int64_t timeout_us) {
  if (pool == nullptr || timeout_us < 0) return SCOUT_ERR_INVALID_ARG;
  std::unique_lock<std::mutex> lk(pool->mu);
  const bool done = pool->cv_done.wait_for(lk, std::chrono::microseconds(timeout_us), [&] { return !pool->running; });
  return done ? SCOUT_OK : SCOUT_ERR_TIMEOUT;
}
