// pa_grid_reduce.cuh -- V2 pass 2 run by the pass-1 grid itself, after its
// streaming, so that the whole V2 step is one launch.
//
// Every CTA streams its work items as usual (each partition's partial written
// to the workspace as the pages' Phase 1 defines it), then counts itself
// finished.  A CTA that finishes after every CTA of the grid has started
// takes reduce units from a queue, waits until every CTA has finished, and
// reduces its units: unit u is (sequence b, query head h, 32-element slice of
// head_dim), computed as
//   M = max_p m_p,  w_p = s_p exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p
// over the row's partitions p < ceil(L_b / P) -- Phase 2 of commit 4eb83a7e
// "qwen3_6_scripts", paragraph "Implementation (paged_attention_v2_pytorch.py)"
// (global max, rescale exp(m_p - global_max) * exp_sum_p, weighted sum over
// the total).  The CTA's four softmax warps (128 threads) share a unit:
// thread t takes float4 column t % 8 of the slice and partitions t / 8,
// t / 8 + 16, ...; the sums are combined in a fixed order, so results are
// bit-identical from run to run.
//
// The reduce runs once per CTA, at the very end of a long kernel, so its code
// would be fetched cold (measured: about 2.7 us of a 3.9 us unit on GB300).
// The standard-layout kernel's softmax warps therefore run the unit once at
// the kernel's start, in a dry mode with no side effects, while the first
// keys are still landing, so that the code is in the SM's instruction cache
// when it is needed.
//
// Forward progress.  Only CTAs that have started can be waited for: a CTA
// waits for the others only if the start counter shows that every CTA of the
// grid has started (so all of them are resident and will finish: no CTA ever
// waits for work of a CTA that has not started).  A CTA that finishes while
// some have not started leaves the reduce to the later ones; the last CTA to
// start always takes part, so every unit is reduced.  Every wait is bounded.
//
// Memory ordering is the grid-barrier pattern: the CTA's threads store their
// partials and meet at a CTA barrier; one thread makes a GPU-scope fence and
// counts the CTA finished; a waiting CTA reads the count, fences, meets its
// threads at a CTA barrier, and they read the partials through L2.
//
// State in the workspace's control block (pa_internal.h), no reset on the
// critical path: the start word holds (launch epoch << 32 | CTAs started);
// the CTA that starts last moves it to (epoch + 1, 0) for the next launch.
// The finished counter and the unit queue come in two banks picked by the
// epoch's parity; the CTA that starts first zeroes the other bank, which
// the previous launch used and the next launch will.
#pragma once

#include <cstddef>
#include <cstdint>

#include "pa_device.cuh"
#include "pa_sm100.cuh"

namespace pa {
namespace gridred {

constexpr int kThreads = 128;                 // the four softmax warps
constexpr int kWarps = kThreads / 32;
constexpr int kSlice = 32;                    // head_dim elements per unit
constexpr int kCols = kSlice / 4;             // float4 columns per unit
constexpr int kLanes = kThreads / kCols;      // partition lanes per column (16)
constexpr int kBoxP = 256;                    // partitions per tile copy (the box's rows)
constexpr int kMaxStats = 1024;               // partitions whose statistics a unit holds

// Control block words (after the status word and the marker).
struct Sync {
  unsigned long long start;  // epoch << 32 | CTAs started
  uint32_t finished[2];      // CTAs finished, by epoch parity
  uint32_t queue[2];         // next reduce unit, by epoch parity
};

__device__ __forceinline__ Sync* sync_words(const KernelArgs& a) {
  return reinterpret_cast<Sync*>(reinterpret_cast<char*>(a.status) + kSyncOffset);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// release: this thread's earlier writes, and those ordered before it by a CTA
// barrier, are visible to whoever acquires the count
__device__ __forceinline__ void red_add_release(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// the softmax warps' named barrier (128 threads)
__device__ __forceinline__ void sync128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Called by one thread at the CTA's start: counts it started and returns the
// start word as it was (epoch, and how many CTAs had started before).
__device__ __forceinline__ unsigned long long count_started(const KernelArgs& a) {
  return atomicAdd(&sync_words(a)->start, 1ull);
}

// Shared scratch of one unit: the small per-warp sums first, then the
// statistics (then the weights), then the tile of partial outputs -- so the
// dry run touches only the first few KB.
struct UnitScratch {
  float4 acc[kWarps][kCols];
  float wsum[kWarps];
  float wmax[kWarps];
  int wnan[kWarps];
  float m[kMaxStats];          // m_p
  float s[kMaxStats];          // s_p, then the weight w_p = s_p exp(m_p - M)
  // o_p[d0 .. d0 + 32) of partitions p0 .. p0 + kBoxP: a tile copy's
  // destination, which must start on a 128-byte boundary
  alignas(128) float4 tile[kBoxP][kCols];
};
static_assert(offsetof(UnitScratch, tile) % 128 == 0, "tile copy destination alignment");
// bytes of the scratch a dry run touches (one partition)
constexpr size_t kDryBytes = offsetof(UnitScratch, tile) + kCols * 16;

// Reduce unit u (the 128 softmax threads) in the order of the pages' Phase 2:
// the row's global max M over its partitions' m_p, the weights
// w_p = s_p exp(m_p - M) (one exp per partition), then out = sum w_p o_p /
// sum w_p, the sums in a fixed order.  Rows of sequences that pass 1 finished
// itself (1..P tokens) are skipped; a sequence of length 0 gets zeros and one
// of invalid length NaN.  With `poison` (the partials cannot be trusted)
// every row the unit would reduce or fill is written as NaN instead.  The
// partial outputs come in by one tile copy per kBoxP partitions (`pmap`:
// tmp_output as [rows][NP][head_dim] floats, box 32 x kBoxP x 1) landing on
// `bar`, whose phase the caller tracks; `L` is the sequence's length.
// `dry`: run the same code over one partition of row 0 with no tile copy and
// no store (only to bring the code into the instruction cache) -- the same
// code, hence out of line: both calls run one copy of it.
template <int D>
__device__ __noinline__ void reduce_unit(const KernelArgs& a, const CUtensorMap* pmap, uint64_t* bar,
                            uint32_t& phase, int64_t u, int32_t L, UnitScratch& sc, int tid,
                            bool poison, long long budget, bool dry) {
  constexpr int kSlices = D / kSlice;
  const int64_t row = u / kSlices;
  const int d0 = static_cast<int>(u % kSlices) * kSlice;
  const int col = tid % kCols, lane = tid / kCols, wp = tid / 32;
  if (!dry) {
    if (seq_len_ok(a, L) && L >= 1 && L <= a.partition_size) return;  // finished in pass 1
    if (poison || !seq_len_ok(a, L) || L == 0) {
      const float v = L == 0 && !poison ? 0.f : qnan();
      if (tid < kCols)
        store_out4(a.out, row * D + d0 + 4 * tid, a.out_dtype, make_float4(v, v, v, v));
      return;
    }
  }
  // <= kMaxStats (host check)
  const int n = dry ? 1 : (L + a.partition_size - 1) / a.partition_size;
  const int64_t NP = a.num_partitions;
  const int boxp = dry ? 1 : static_cast<int>(NP < kBoxP ? NP : kBoxP);
  if (tid == 0 && !dry) {  // the first tile copy flies while the statistics are read
    sm100::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kSlice * boxp * 4));
    sm100::tma_load_3d(&sc.tile[0][0], pmap, bar, d0, 0, static_cast<int32_t>(row),
                       sm100::l2_evict_first_policy());
  }
  // M = max m_p, and whether any m_p is NaN (a poisoned partition)
  const float* ml = a.max_logits + row * NP;
  const float* es = a.exp_sums + row * NP;
  float mx = -INFINITY;
  bool nan = false;
  for (int i = tid; i < n; i += kThreads) {
    const float m = __ldcg(ml + i);
    sc.m[i] = m;
    sc.s[i] = __ldcg(es + i);
    nan |= isnan(m);
    mx = fmaxf(mx, m);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  nan = __any_sync(0xffffffffu, nan);
  if ((tid & 31) == 0) {
    sc.wmax[wp] = mx;
    sc.wnan[wp] = nan ? 1 : 0;
  }
  sync128();
  float M = sc.wmax[0];
  bool bad = sc.wnan[0] != 0;
#pragma unroll
  for (int k = 1; k < kWarps; ++k) {
    M = fmaxf(M, sc.wmax[k]);
    bad |= sc.wnan[k] != 0;
  }
  // the weights, one exp per partition
  for (int i = tid; i < n; i += kThreads) {
    const float m = sc.m[i];
    sc.s[i] = m == -INFINITY ? 0.f : sc.s[i] * expf(m - M);
  }
  sync128();
  float W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p0 = 0; p0 < n; p0 += boxp) {
    const int cnt = min(boxp, n - p0);
    if (!dry) {
      if (p0 > 0 && tid == 0) {
        sm100::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kSlice * boxp * 4));
        sm100::tma_load_3d(&sc.tile[0][0], pmap, bar, d0, p0, static_cast<int32_t>(row),
                           sm100::l2_evict_first_policy());
      }
      if (!sm100::mbar_wait(bar, phase, budget, nullptr)) {
        set_status(a.status, PA_ERR_DEVICE_TIMEOUT);
        bad = true;
        sm100::mbar_wait(bar, phase, budget, nullptr);  // the copy lands before reuse
      }
      phase ^= 1u;
    }
    for (int i = lane; i < cnt; i += kLanes) {
      const float e = sc.s[p0 + i];
      const float4 o = sc.tile[i][col];
      W += e;
      acc.x = fmaf(e, o.x, acc.x);
      acc.y = fmaf(e, o.y, acc.y);
      acc.z = fmaf(e, o.z, acc.z);
      acc.w = fmaf(e, o.w, acc.w);
    }
    sync128();  // the tile may be overwritten
  }
  // sum over the lanes of each column: within a warp, then the warps in order
#pragma unroll
  for (int off = kCols; off < 32; off <<= 1) {
    W += __shfl_xor_sync(0xffffffffu, W, off);
    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
  }
  if ((tid & 31) < kCols) {
    sc.acc[wp][col] = acc;
    if (col == 0) sc.wsum[wp] = W;
  }
  sync128();
  if (tid < kCols) {
    float4 S = sc.acc[0][tid];
    float T = sc.wsum[0];
#pragma unroll
    for (int k = 1; k < kWarps; ++k) {
      const float4 v = sc.acc[k][tid];
      S.x += v.x;
      S.y += v.y;
      S.z += v.z;
      S.w += v.w;
      T += sc.wsum[k];
    }
    const float4 r = bad ? make_float4(qnan(), qnan(), qnan(), qnan())
                         : make_float4(S.x / T, S.y / T, S.z / T, S.w / T);
    if (!dry) store_out4(a.out, row * D + d0 + 4 * tid, a.out_dtype, r);
  }
  sync128();  // the scratch may be reused
}

// The end of a one-launch V2 grid, run by the 128 softmax threads after the
// CTA's streaming (with a CTA barrier after its last partial store): count
// the CTA finished, and if every CTA has started, reduce units from the queue
// once every CTA has finished.  `ws_ok`: the workspace carries the
// initialisation marker (else no counter is touched and the rows that needed
// pass 2 become NaN, split statically over the CTAs).  `started` is thread
// 0's count_started() result; `w` three shared ints for broadcasts; `sc` the
// unit's shared scratch; `pmap` / `bar`: the tile copy of the partials and
// its mbarrier (initialised, phase 0).  `dry`: the same code with no effect
// (counts of 0, one poll, no unit), run at the kernel's start so that the
// code is in the instruction cache at the end -- hence out of line.
template <int D>
__device__ __noinline__ void grid_reduce(const KernelArgs& a, bool ws_ok,
                                         unsigned long long started, int* w, UnitScratch& sc,
                                         const CUtensorMap* pmap, uint64_t* bar, int tid,
                                         long long budget, bool dry) {
  constexpr int kSlices = D / kSlice;
  const int64_t units = static_cast<int64_t>(a.num_seqs) * a.num_heads * kSlices;
  auto seq_len_of = [&](int64_t u) { return __ldg(a.seq_lens + u / kSlices / a.num_heads); };
  uint32_t phase = 0;
  if (!ws_ok) {
    for (int64_t u = blockIdx.x; u < units && !dry; u += gridDim.x)
      reduce_unit<D>(a, pmap, bar, phase, u, seq_len_of(u), sc, tid, true, budget, false);
    return;
  }
  Sync* s = sync_words(a);
  const uint32_t grid = gridDim.x;
  const uint32_t epoch = static_cast<uint32_t>(started >> 32);
  const int bank = epoch & 1;
  const uint32_t one = dry ? 0u : 1u;
  if (tid == 0) {
    const uint32_t rank = static_cast<uint32_t>(started);
    red_add_release(&s->finished[bank], one);  // every thread's partials precede the count
    if (rank == 0 && !dry) {  // the other bank: used by the last launch, next by the next one
      s->finished[bank ^ 1] = 0u;
      s->queue[bank ^ 1] = 0u;
    }
    if (rank == grid - 1 && !dry)  // the last CTA to start: the next launch's epoch
      red_add64(&s->start, (1ull << 32) - grid);
    // every CTA has started when the count is complete or the epoch moved on
    const unsigned long long now = ld_relaxed64(&s->start);
    const bool all = static_cast<uint32_t>(now >> 32) != epoch ||
                     static_cast<uint32_t>(now) >= grid;
    int unit = static_cast<int>(units);  // none
    int timed_out = 0;
    int32_t L = 0;
    if (all || dry) {
      const int got = static_cast<int>(atomicAdd(&s->queue[bank], one));
      if (!dry) unit = got;
      if (unit < units || dry) {
        L = seq_len_of(dry ? 0 : unit);  // an input: read while the others finish
        const long long t0 = clock64();
        while (ld_acquire(&s->finished[bank]) < grid) {  // every CTA's partials stored
          if (dry) break;
          if (clock64() - t0 > budget) {
            set_status(a.status, PA_ERR_DEVICE_TIMEOUT);
            timed_out = 1;  // this CTA's units are written as NaN
            break;
          }
          __nanosleep(64);
        }
      }
    }
    w[0] = unit;
    w[1] = timed_out;
    w[2] = L;
  }
  sync128();
  int unit = w[0];
  int32_t L = w[2];
  const bool poison = w[1] != 0;
  while (unit < units) {
    reduce_unit<D>(a, pmap, bar, phase, unit, L, sc, tid, poison, budget, false);
    if (tid == 0) {
      w[0] = static_cast<int>(atomicAdd(&s->queue[bank], 1u));
      if (w[0] < units) w[2] = seq_len_of(w[0]);
    }
    sync128();
    unit = w[0];
    L = w[2];
    sync128();  // every thread has read w[] before thread 0 writes it again
  }
}

}  // namespace gridred
}  // namespace pa
