// pa_sx.cuh -- tensor-core decode kernel for caches in the split-x layout.
//
// The layout commit 4eb83a7e "qwen3_6_scripts", paragraph "Hardware testing
// confirmed", gives for its V1 kernel:
//   keys   [blocks, kv_heads, head_dim / x, block_size, x]  (x = 8 for 16-bit)
//   values [blocks, kv_heads, head_dim, block_size]
// One (block, KV head) of either cache is one contiguous region of
// block_size * head_dim elements, so a block comes in by two bulk copies
// (cp.async.bulk, 8 KB each for 16 tokens of head_dim 256).  The shared-memory
// descriptors of tcgen05.mma need 8-row groups at one uniform stride, which
// blocks scattered over the pool do not give; the warp-level MMA
// (mma.sync.m16n8k16) takes its operands from registers, loaded with ldmatrix
// from any eight 16-byte rows, and a split-x key group is exactly such a set
// of rows (8 consecutive head_dim elements of one token per row), as is a
// transposed value row (8 consecutive tokens of one head_dim element).  The
// kernel is bound by HBM, not by the tensor pipe.
//
// Work item: one (sequence, KV head, token range), the range a V2 partition
// or the whole sequence (V1); the G <= 8 query heads of the KV head are
// served together.  The grid is persistent (at most two CTAs per SM, the
// items dealt out in balanced rounds): CTA c takes items c, c + gridDim.x,
// ...; with fewer items than SMs, a cluster of up to 16 CTAs shares each
// item instead (each CTA a balanced run of its chunks) and the CTAs merge
// their partial results through distributed shared memory at the end.
// Warp 4 streams the blocks of all its items, one after the other, into
// one ring of whole blocks (keys and values), so the next item's blocks are
// in flight while the current one finishes, and loads each item's q rows by
// bulk copy into one of two q tiles; warps 0-3 consume the ring in chunks of
// 32 tokens at head_dim 256 (64 at 128, 128 at 64: the same bytes):
//   QK^T   warp w: S[h, t] for its quarter of the chunk, in n-tiles of 8
//          tokens, over all of head_dim (A = q, rows 0..7 = the query
//          heads; B = keys);
//   softmax the chunk's max per head across the four warps (shared memory),
//          p = exp2(l - m), the running max / sum / rescale across chunks;
//   P.V    warp w: head_dim slice w of O[h, d] over the chunk's tokens;
//          A = P with rows 0..7 its 16-bit hi part and rows 8..15 the
//          rounded remainder, so one MMA carries ~16 significant bits of p
//          and O = (rows 0..7) + (rows 8..15) at the end.
// Logits are f32 sums of exact 16-bit products, scaled into base 2 after.
//
// This is Phase 1 of the V2 scheme of commit 4eb83a7e "qwen3_6_scripts",
// paragraph "Implementation (paged_attention_v2_pytorch.py)", or V1 when the
// range is the whole sequence.  With a.fused the same grid then runs Phase 2
// (the grid-end reduce of pa_grid_reduce.cuh, by the four consumer warps,
// scratch in the ring), so the V2 step is one launch.  Every wait is
// bounded; a wait that gives up sets PA_ERR_DEVICE_TIMEOUT and the item's
// outputs become NaN.
#pragma once

#include <algorithm>
#include <atomic>
#include <type_traits>

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_grid_reduce.cuh"
#include "pa_sm100.cuh"

namespace pa {
namespace sx {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
// Tokens per chunk: 8 per consumer warp and n-tile of QK^T, with more
// n-tiles per warp for smaller head_dim, so that a chunk carries as many
// bytes (and amortises its barriers as well) at every head_dim
template <int D>
constexpr int chunk_tokens() { return D >= 256 ? 32 : (D == 128 ? 64 : 128); }
constexpr int kRingBytes = 96 * 1024;                // two CTAs per SM
constexpr int kMaxStages = 24;
constexpr long long kWaitBudget = 4000000000LL;      // cycles (about 2 s)
constexpr long long kSelftestBudget = 20000000LL;    // cycles (about 10 ms)

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}

// D (16 x 8, f32) += A (16 x 16) * B (16 x 8), 16-bit inputs.
template <typename T>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to shared memory, counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(sm100::smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(sm100::smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// consumer_sync that also returns whether any consumer thread passed true
__device__ __forceinline__ bool consumer_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.or.pred q, 1, 128, p;\n"
      "selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}

// Two 16-bit values in one register (low half: the first).
template <typename T>
__device__ __forceinline__ uint32_t pack2(T lo, T hi) {
  return static_cast<uint32_t>(bits16(lo)) | (static_cast<uint32_t>(bits16(hi)) << 16);
}

constexpr int kQRows = 8;  // q tile rows: the query heads of one KV head
constexpr int kMaxCompactSeqs = 1024;  // V2 batches up to this size walk a compact list
// A cluster share's partial at the start of the ring (floats): per head m
// and s, a poison flag, then O [8 heads][head_dim] (unnormalised)
constexpr int kMergeM = 0, kMergeS = 8, kMergePoison = 16, kMergeO = 32;

template <int D, int BS>
struct Layout {
  static constexpr int kBlockBytes = BS * D * 2;            // one block of one cache
  static constexpr int kStageBytes = 2 * kBlockBytes;       // keys + values
  static constexpr int kStages =
      kRingBytes / kStageBytes < kMaxStages ? kRingBytes / kStageBytes : kMaxStages;
  static constexpr int kChunk = chunk_tokens<D>();
  static constexpr int kNT = kChunk / 32;                    // QK^T n-tiles per warp
  static constexpr int kChunkBlocks = kChunk / BS > 0 ? kChunk / BS : 1;
  static constexpr int kQStride = D + 8;                     // q tile row (elements), padded
  static constexpr int kQTile = kQRows * kQStride;           // elements of one q tile
  static constexpr int kPStride = kChunk + 8;                // P tile row (elements), padded
  static constexpr int kQOff = kStages * kStageBytes;        // two q tiles
  static constexpr int kPOff = kQOff + 2 * kQTile * 2;
  static constexpr int kRedOff = kPOff + 16 * kPStride * 2;  // [4 warps][8 heads] max, sum
  static constexpr int kBarOff = kRedOff + 2 * kConsumerWarps * 8 * 4;
  // full[kMaxStages], empty[kMaxStages], qfull[2], qempty[2], for the
  // one-launch V2 grid red_bar (a reduce unit's tile copy), and never (the
  // self-test's wait: nothing arrives there)
  static constexpr int kFlagOff = kBarOff + (2 * kMaxStages + 6) * 8;
  // [0] abort; [1 + s] ring slot s holds no block (its id was out of range);
  // [kWsOk] the workspace carries the init marker; [kRedWord ..] three ints
  // for the reduce's broadcasts
  static constexpr int kWsOk = 1 + kMaxStages;
  static constexpr int kRedWord = kWsOk + 1;
  static constexpr int kScan = kRedWord + 3;       // [kThreads / 32] warp totals
  static constexpr int kTotalOff = (kFlagOff + (kScan + 8) * 4 + 7) / 8 * 8;  // int64 items
  // compact work list (V2, 2..kMaxCompactSeqs sequences): prefix[b] =
  // partitions of the sequences before b
  static constexpr int kPrefixOff = kTotalOff + 8;
  static constexpr int kSmem = kPrefixOff + (kMaxCompactSeqs + 1) * 4 + 64;
  // One-launch V2: the reduce's scratch is the ring once streaming is done.
  // (No dry run of the reduce at the start, unlike the standard-layout
  // kernel: here it would hold back the first fill of the ring slots it
  // borrows, which measured 2.4 us slower per step than the cold code it
  // saves at the end.)
  static_assert(sizeof(gridred::UnitScratch) <= kStages * kStageBytes, "reduce scratch in the ring");
  static_assert(kStages >= 2 * kChunkBlocks, "two chunks in flight");
  static_assert((kQStride * 2) % 16 == 0 && kQOff % 16 == 0, "bulk copies of q rows");
  static_assert(kSmem <= 113 * 1024, "two CTAs per SM");
};

// One work item, decoded the same way by the producer and the consumers.
struct Item {
  int b, kvh, part;
  int32_t t0, t1;  // token range (empty when t0 >= t1)
  bool len_ok;     // 0 <= seq_len <= max_seq_len
  bool direct;     // V2 with single_direct: the result is the final output
  bool any;        // the item's whole range (over all CTAs of a cluster) has tokens
  int nblk;        // blocks of this CTA's range (0 when it is empty)
};

// Item k of the (partition, sequence, KV head) space, partition-major for V2
// (ranges past a sequence's end come out empty), (sequence, KV head) for V1.
// With a cluster of cs CTAs sharing the item, CTA `rank` takes a balanced
// run of its kChunk-token chunks.
// With a compact work list (`prefix`, V2) k runs over the (sequence,
// partition, KV head) triples that exist, sequence-major.
template <int BS, int kChunk>
__device__ __forceinline__ Item item_at(const KernelArgs& a, const int32_t* prefix, int64_t k,
                                        bool v2, int rank, int cs) {
  Item it;
  if (prefix) {
    const int64_t j = k / a.num_kv_heads;
    it.kvh = static_cast<int>(k % a.num_kv_heads);
    int lo = 0, hi = a.num_seqs;  // largest lo with prefix[lo] <= j
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= j) lo = mid;
      else hi = mid;
    }
    it.b = lo;
    it.part = static_cast<int>(j - prefix[lo]);
  } else {
    const int64_t per_part = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads;
    it.part = v2 ? static_cast<int>(k / per_part) : 0;
    const int64_t rem = v2 ? k % per_part : k;
    it.b = static_cast<int>(rem / a.num_kv_heads);
    it.kvh = static_cast<int>(rem % a.num_kv_heads);
  }
  const int32_t L = __ldg(a.seq_lens + it.b);
  it.len_ok = seq_len_ok(a, L);
  it.t0 = v2 ? it.part * a.partition_size : 0;  // a multiple of BS
  it.t1 = !it.len_ok ? it.t0 : (v2 ? min(L, it.t0 + a.partition_size) : L);
  it.direct = v2 && a.single_direct && it.len_ok && L <= a.partition_size;
  it.any = it.t0 < it.t1;
  if (cs > 1 && it.any) {
    const int nch = (it.t1 - it.t0 + kChunk - 1) / kChunk;
    const int lo = rank * nch / cs, hi = (rank + 1) * nch / cs;
    it.t1 = min(it.t1, it.t0 + hi * kChunk);
    it.t0 += lo * kChunk;  // a multiple of kChunk, so of BS; empty when lo == hi
  }
  it.nblk = it.t0 < it.t1 ? (it.t1 - 1) / BS - it.t0 / BS + 1 : 0;
  return it;
}

}  // namespace sx

template <typename T, int D, int BS, bool kV2>
__global__ void __launch_bounds__(sx::kThreads, 2)
    pa_sx_kernel(const KernelArgs a, const __grid_constant__ CUtensorMap pmap, int64_t grid_items,
                 int compact, int cs) {
  using namespace sx;
  using Lay = Layout<D, BS>;
  static_assert(BS == 16 || BS == 32, "block size");
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  T* qs = reinterpret_cast<T*>(smem + Lay::kQOff);  // two tiles of kQRows x kQStride
  T* ps = reinterpret_cast<T*>(smem + Lay::kPOff);
  float* red_max = reinterpret_cast<float*>(smem + Lay::kRedOff);
  float* red_sum = red_max + kConsumerWarps * 8;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lay::kBarOff);
  uint64_t* empty = full + kMaxStages;
  uint64_t* qfull = empty + kMaxStages;
  uint64_t* qempty = qfull + 2;
  uint64_t* red_bar = qempty + 2;
  uint64_t* never = red_bar + 1;
  int* flags = reinterpret_cast<int*>(smem + Lay::kFlagOff);
  volatile int* abort_flag = &flags[0];
  volatile int* bad = flags + 1;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.group, Hq = a.num_heads;
  const T zero = round16(0.f, static_cast<T*>(nullptr));
  // Clusters of cs CTAs (cs == 1: none) share each work item: the host then
  // launches one cluster per item, and CTA `rank` streams its share.
  const int rank = cs > 1 ? static_cast<int>(blockIdx.x % cs) : 0;
  const int64_t cid = blockIdx.x / cs, cstride = gridDim.x / cs;

  // ---- set-up ---------------------------------------------------------------------
  const bool fused = kV2 && a.fused;  // one-launch V2: pass 2 by this grid at the end
  unsigned long long started = 0;     // thread 0, one-launch V2: the start word as it was
  if (tid == 0) {
    for (int s = 0; s < Lay::kStages; ++s) {
      sm100::mbar_init(&full[s], 1);
      sm100::mbar_init(&empty[s], kConsumerWarps);
      bad[s] = 0;
    }
    for (int i = 0; i < 2; ++i) {
      sm100::mbar_init(&qfull[i], 1);
      sm100::mbar_init(&qempty[i], kConsumerWarps);
    }
    sm100::mbar_init(never, 1);
    flags[0] = 0;
    // one-launch V2: the counters are usable only in an initialised workspace;
    // the CTA counts itself started (the result is first used at the end)
    int ws_ok = 0;
    if (fused) {
      sm100::mbar_init(red_bar, 1);
      ws_ok = __ldcg(a.status + kMarkerOffset / 4) == kMarker;
      if (ws_ok)
        started = gridred::count_started(a);
      else
        set_status(a.status, PA_ERR_WORKSPACE_NOT_INIT);
    }
    flags[Lay::kWsOk] = ws_ok;
  }
  // rows G .. 7 of both q tiles stay zero; the bulk copies fill rows 0 .. G-1
  for (int i = tid; i < 2 * kQRows * D; i += kThreads) {
    const int r = (i / D) % kQRows, tile = i / (kQRows * D);
    if (r >= G) qs[tile * Lay::kQTile + r * Lay::kQStride + i % D] = zero;
  }
  int32_t* const prefix_s = reinterpret_cast<int32_t*>(smem + Lay::kPrefixOff);
  int64_t* const total_s = reinterpret_cast<int64_t*>(smem + Lay::kTotalOff);
  if (compact) {
    // Compact work list: prefix[b] = partitions of the sequences before b.
    // A sequence whose length is outside 0..max_seq_len contributes none
    // (the reduce writes its NaN rows).
    int* const scan = flags + Lay::kScan;
    int carry = 0;
    for (int base = 0; base < a.num_seqs; base += kThreads) {
      const int b = base + tid;
      int n = 0;
      if (b < a.num_seqs) {
        const int32_t L = __ldg(a.seq_lens + b);
        if (seq_len_ok(a, L))
          n = (L + a.partition_size - 1) / a.partition_size;
        else if (blockIdx.x == 0)
          set_status(a.status, PA_ERR_BAD_SEQ_LEN);
      }
      int x = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) scan[warp] = x;
      __syncthreads();
      int off = 0, round_total = 0;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) {
        off += w < warp ? scan[w] : 0;
        round_total += scan[w];
      }
      if (b < a.num_seqs) prefix_s[b + 1] = carry + off + x;
      carry += round_total;
      __syncthreads();
    }
    if (tid == 0) {
      prefix_s[0] = 0;
      *total_s = static_cast<int64_t>(carry) * a.num_kv_heads;
    }
  } else if (tid == 0) {
    *total_s = grid_items;
  }
  __syncthreads();
  const int32_t* const prefix = compact ? prefix_s : nullptr;
  const int64_t total_items = *total_s;

  if (warp == kConsumerWarps) {
    // ========================= producer =======================================
    const uint64_t policy = sm100::l2_evict_first_policy();
    const uint64_t qpolicy = sm100::l2_evict_last_policy();  // q: read once per partition
    const char* kc = static_cast<const char*>(a.k_cache);
    const char* vc = static_cast<const char*>(a.v_cache);
    const char* qg = static_cast<const char*>(a.q);
    if (fused && lane == 0) sm100::tma_prefetch_desc(&pmap);
    bool ok = true;
    // self-test (PA_FLAG_SELFTEST_STALL): a wait that runs out, so that the
    // abort path runs (no copy issued; every output of the call becomes NaN)
    if (a.selftest_stall)
      ok = __all_sync(0xffffffffu, sm100::mbar_wait(never, 0, kSelftestBudget, abort_flag));
    uint32_t jg = 0;  // ring blocks issued, over all items (a CTA streams far
                      // fewer than 2^32 blocks, so 32 bits keep the slot
                      // arithmetic short)
    int nq = 0;      // q tiles issued
    for (int64_t k = cid; k < total_items && ok; k += cstride) {
      const Item it = item_at<BS, Lay::kChunk>(a, prefix, k, kV2, rank, cs);
      if (it.nblk == 0) continue;
      const int qb = nq & 1;
      ok = __all_sync(0xffffffffu, sm100::mbar_wait(&qempty[qb], ((nq >> 1) & 1) ^ 1,
                                                    kWaitBudget, abort_flag));
      if (!ok) break;
      if (lane == 0) {
        const int64_t row0 = static_cast<int64_t>(it.b) * Hq + static_cast<int64_t>(it.kvh) * G;
        sm100::mbar_arrive_expect_tx(&qfull[qb], G * D * 2);
        for (int r = 0; r < G; ++r)
          bulk_g2s(qs + qb * Lay::kQTile + r * Lay::kQStride, qg + (row0 + r) * D * 2, D * 2,
                   &qfull[qb], qpolicy);
      }
      __syncwarp();
      ++nq;
      const int32_t* bt =
          a.block_tables + static_cast<int64_t>(it.b) * a.max_blocks_per_seq + it.t0 / BS;
      for (int j0 = 0; j0 < it.nblk && ok; j0 += 32) {
        const int32_t id_l = j0 + lane < it.nblk ? __ldg(bt + j0 + lane) : 0;
        const int n32 = min(32, it.nblk - j0);
        for (int jj = 0; jj < n32; ++jj, ++jg) {
          const int slot = static_cast<int>(jg % Lay::kStages);
          const uint32_t par = static_cast<uint32_t>((jg / Lay::kStages) & 1) ^ 1;
          ok = __all_sync(0xffffffffu,
                          sm100::mbar_wait(&empty[slot], par, kWaitBudget, abort_flag));
          if (!ok) break;
          const int32_t id = __shfl_sync(0xffffffffu, id_l, jj);
          if (lane == 0) {
            if (id < 0 || id >= a.num_blocks) {  // never read: the item becomes NaN
              bad[slot] = 1;
              set_status(a.status, PA_ERR_BAD_BLOCK_ID);
              sm100::mbar_arrive(&full[slot]);
            } else {
              bad[slot] = 0;
              const int64_t off =
                  (static_cast<int64_t>(id) * a.num_kv_heads + it.kvh) * Lay::kBlockBytes;
              uint8_t* st = ring + slot * Lay::kStageBytes;
              sm100::mbar_arrive_expect_tx(&full[slot], Lay::kStageBytes);
              bulk_g2s(st, kc + off, Lay::kBlockBytes, &full[slot], policy);
              bulk_g2s(st + Lay::kBlockBytes, vc + off, Lay::kBlockBytes, &full[slot], policy);
            }
          }
          __syncwarp();
        }
      }
    }
    if (!ok) {
      if (lane == 0) {
        flags[0] = 1;
        set_status(a.status, PA_ERR_DEVICE_TIMEOUT);
      }
      // copies issued must land before the CTA may exit
      for (uint32_t j = jg > Lay::kStages ? jg - Lay::kStages : 0; j < jg; ++j)
        sm100::mbar_wait(&full[j % Lay::kStages], static_cast<uint32_t>((j / Lay::kStages) & 1),
                         kWaitBudget, nullptr);
      for (int i = nq > 2 ? nq - 2 : 0; i < nq; ++i)
        sm100::mbar_wait(&qfull[i & 1], (i >> 1) & 1, kWaitBudget, nullptr);
    }
    if (cs == 1) return;  // in a cluster the warp meets the merge's barriers below
  } else {
  // =========================== consumers (warps 0-3) ================================
  const int g = lane >> 2, t = lane & 3;  // mma fragment: row group, column pair
  const float sl2 = a.scale_log2;
  const uint32_t p_base = sm100::smem_u32(ps);
  const uint32_t ring_base = sm100::smem_u32(ring);
  constexpr int kDT = D / 4 / 8;  // 8-wide head_dim tiles of this warp's P.V slice
  // a cluster share's result, left for the merge at the start of the ring
  // (every block of the share was consumed: the ring is free)
  float* const mgp = reinterpret_cast<float*>(ring);
  auto write_partial = [&](float m, float sv, float (*accp)[kDT][4], bool pois) {
    const bool any_pois = consumer_any(pois);  // a barrier too: the ring reads are done
    if (g < G) {
#pragma unroll
      for (int i = 0; i < kDT; ++i) {
        const int d = warp * (D / 4) + i * 8 + 2 * t;
        mgp[kMergeO + g * D + d] = accp ? (*accp)[i][0] + (*accp)[i][2] : 0.f;
        mgp[kMergeO + g * D + d + 1] = accp ? (*accp)[i][1] + (*accp)[i][3] : 0.f;
      }
      if (warp == 0 && t == 0) {
        mgp[kMergeM + g] = m;
        mgp[kMergeS + g] = sv;
      }
    }
    if (tid == 0) mgp[kMergePoison] = any_pois ? 1.f : 0.f;
  };
  int hs = 0;                      // ring slot of the next block to consume
  uint32_t hp = 0;                 // and its phase parity (no division in the hot loop)
  auto wrap = [](int x) { return x >= Lay::kStages ? x - Lay::kStages : x; };
  int nq = 0;                     // q tiles consumed
  int* const red_word = flags + Lay::kRedWord;
  for (int64_t k = cid; k < total_items; k += cstride) {
    const Item it = item_at<BS, Lay::kChunk>(a, prefix, k, kV2, rank, cs);
    const int64_t row0 = static_cast<int64_t>(it.b) * Hq + static_cast<int64_t>(it.kvh) * G;
    if (it.nblk == 0) {
      if (!it.len_ok && tid == 0 && it.part == 0 && rank == 0)
        set_status(a.status, PA_ERR_BAD_SEQ_LEN);
      if (cs > 1) {  // an empty share: the merge sees m = -inf, s = 0, O = 0
        write_partial(-INFINITY, 0.f, nullptr, false);
        continue;
      }
      if (!kV2) {  // V1: NaN rows for a bad length, zero rows for an empty sequence
        const float v = it.len_ok ? 0.f : qnan();
        for (int i = tid; i < G * D; i += kConsumerWarps * 32)
          store_out(a.out, row0 * D + i, a.out_dtype, v);
      }
      continue;  // V2: the reduce writes those rows
    }
    const int qb = nq & 1;
    bool poison = false;
    if (!sm100::mbar_wait(&qfull[qb], (nq >> 1) & 1, kWaitBudget, abort_flag)) {
      poison = true;
      if (lane == 0) {
        flags[0] = 1;
        set_status(a.status, PA_ERR_DEVICE_TIMEOUT);
      }
    }
    // q as A fragments for the whole item: rows 0..7 the query heads (rows
    // 8..15 of the MMA are zero), qf[ks] = columns 16 ks .. 16 ks + 15
    uint32_t qf[D / 16][2];
    {
      const uint32_t q_base = sm100::smem_u32(qs + qb * Lay::kQTile);
#pragma unroll
      for (int ks = 0; ks < D / 16; ks += 2) {
        uint32_t r[4];
        ldsm_x4(r, q_base + ((lane & 7) * Lay::kQStride + ks * 16 + (lane >> 3) * 8) * 2);
        qf[ks][0] = r[0];
        qf[ks][1] = r[1];
        qf[ks + 1][0] = r[2];
        qf[ks + 1][1] = r[3];
      }
    }
    float acc[kDT][4];
#pragma unroll
    for (int i = 0; i < kDT; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
    float m_run = -INFINITY, s_run = 0.f;  // for head g (rows g and g + 8)
    const int nchunks = (it.t1 - it.t0 + Lay::kChunk - 1) / Lay::kChunk;
    for (int ci = 0; ci < nchunks; ++ci) {
      const int c0 = it.t0 + ci * Lay::kChunk;
      const int n = min(Lay::kChunk, it.t1 - c0);
      const int nb = (n + BS - 1) / BS;
      // every block of the chunk landed
      for (int i = 0; i < nb; ++i) {
        const int slot = wrap(hs + i);
        if (!sm100::mbar_wait(&full[slot], hs + i >= Lay::kStages ? hp ^ 1u : hp, kWaitBudget,
                              abort_flag)) {
          poison = true;
          if (lane == 0) {
            flags[0] = 1;
            set_status(a.status, PA_ERR_DEVICE_TIMEOUT);
          }
        }
        poison |= bad[slot] != 0;
      }
      // ---- QK^T: this warp's kNT n-tiles of 8 tokens from 8 kNT w ------------------
      constexpr int kNT = Lay::kNT;
      const int tk0 = warp * 8 * kNT;  // first token of this warp's n-tiles in the chunk
      float l[kNT][2];                 // logits of head g, tokens tk + 2t, tk + 2t + 1
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const int tk = tk0 + 8 * nt;
        const int so = tk % BS;
        const uint32_t kblk = ring_base + wrap(hs + tk / BS) * Lay::kStageBytes;
        float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
        if (tk < n) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t kb[2];
            const uint32_t qa[4] = {qf[ks][0], 0u, qf[ks][1], 0u};
            // B: tokens so .. so + 7 of key groups 2 ks and 2 ks + 1 (16 bytes each)
            ldsm_x2(kb, kblk + (((2 * ks + ((lane >> 3) & 1)) * BS + so + (lane & 7)) * 16));
            if (ks & 1) mma16816<T>(sd, qa, kb);  // two chains: half the dependent MMAs
            else mma16816<T>(sc, qa, kb);
          }
        }
        // c[0], c[1]: head g, tokens tk + 2t, tk + 2t + 1; c[2], c[3] are padding
        l[nt][0] = (tk + 2 * t < n && g < G) ? (sc[0] + sd[0]) * sl2 : -INFINITY;
        l[nt][1] = (tk + 2 * t + 1 < n && g < G) ? (sc[1] + sd[1]) * sl2 : -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) mx = fmaxf(mx, fmaxf(l[nt][0], l[nt][1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (t == 0) red_max[warp * 8 + g] = mx;
      consumer_sync();
      float mc = red_max[g];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) mc = fmaxf(mc, red_max[w * 8 + g]);
      const float m_new = fmaxf(m_run, mc);
      float ssum = 0.f;
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
        const float p0 = l[nt][0] == -INFINITY ? 0.f : exp2f(l[nt][0] - m_new);
        const float p1 = l[nt][1] == -INFINITY ? 0.f : exp2f(l[nt][1] - m_new);
        ssum += p0 + p1;
        // P tile: row g = the hi parts, row g + 8 = the remainders
        const int col = tk0 + 8 * nt + 2 * t;
        const T h0 = round16(p0, static_cast<T*>(nullptr)), h1 = round16(p1, static_cast<T*>(nullptr));
        const T r0 = round16(p0 - to_float(h0), static_cast<T*>(nullptr));
        const T r1 = round16(p1 - to_float(h1), static_cast<T*>(nullptr));
        *reinterpret_cast<uint32_t*>(ps + g * Lay::kPStride + col) = pack2<T>(h0, h1);
        *reinterpret_cast<uint32_t*>(ps + (g + 8) * Lay::kPStride + col) = pack2<T>(r0, r1);
      }
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 1);
      ssum += __shfl_xor_sync(0xffffffffu, ssum, 2);
      if (t == 0) red_sum[warp * 8 + g] = ssum;
      // the tail block: value columns past the range are cleared (P is 0 there,
      // but 0 * NaN would be NaN); the slot is refilled by bulk copy later
      if (n < nb * BS) {
        T* vt = reinterpret_cast<T*>(ring + wrap(hs + nb - 1) * Lay::kStageBytes +
                                     Lay::kBlockBytes);
        const int valid = n - (nb - 1) * BS;
        for (int i = tid; i < D * (BS - valid); i += kConsumerWarps * 32) {
          const int d = i / (BS - valid), s = valid + i % (BS - valid);
          vt[d * BS + s] = zero;
        }
        sm100::fence_proxy_async_smem();
      }
      consumer_sync();
      float cs = red_sum[g];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) cs += red_sum[w * 8 + g];
      const float f = m_run == -INFINITY ? 0.f : exp2f(m_run - m_new);
      s_run = s_run * f + cs;
      m_run = m_new;
      // ---- P.V: this warp's head_dim slice over the chunk's tokens ---------------
#pragma unroll
      for (int i = 0; i < kDT; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] *= f;
      for (int kk = 0; kk * 16 < n; ++kk) {  // 16 tokens per step
        uint32_t pa[4];
        ldsm_x4(pa, p_base + (((lane & 7) + ((lane >> 3) & 1) * 8) * Lay::kPStride + kk * 16 +
                              (lane >> 4) * 8) * 2);
        const int sv = (kk * 16) % BS;
        const uint32_t vblk = ring_base +
                              wrap(hs + (kk * 16) / BS) * Lay::kStageBytes + Lay::kBlockBytes;
#pragma unroll
        for (int i = 0; i < kDT; ++i) {
          const int d0 = warp * (D / 4) + i * 8;
          uint32_t vb[2];
          // B: head_dim rows d0 .. d0 + 7, tokens sv + 8 ((lane / 8) % 2) .. + 7
          ldsm_x2(vb, vblk + ((d0 + (lane & 7)) * BS + sv + ((lane >> 3) & 1) * 8) * 2);
          mma16816<T>(acc[i], pa, vb);
        }
      }
      consumer_sync();  // the P tile and the reductions are read before the next chunk
      if (lane == 0)
        for (int i = 0; i < nb; ++i) sm100::mbar_arrive(&empty[wrap(hs + i)]);
      hs += nb;
      if (hs >= Lay::kStages) {
        hs -= Lay::kStages;
        hp ^= 1u;
      }
    }
    ++nq;
    if (lane == 0) sm100::mbar_arrive(&qempty[qb]);  // this item's QK^T is done with q

    // ---- epilogue: O[g] = (rows g + rows g + 8) / s --------------------------------
    poison |= *abort_flag != 0;
    if (cs > 1) {  // the cluster merges the CTAs' shares below
      write_partial(m_run, s_run, &acc, poison);
      continue;
    }
    if (g < G) {
      const int64_t row = row0 + g;
#pragma unroll
      for (int i = 0; i < kDT; ++i) {
        const int d = warp * (D / 4) + i * 8 + 2 * t;
        const float o0 = poison ? qnan() : (acc[i][0] + acc[i][2]) / s_run;
        const float o1 = poison ? qnan() : (acc[i][1] + acc[i][3]) / s_run;
        if (kV2 && !it.direct) {
          float* dst = a.tmp_out + (row * a.num_partitions + it.part) * D + d;
          dst[0] = o0;
          dst[1] = o1;
        } else {
          store_out(a.out, row * D + d, a.out_dtype, o0);
          store_out(a.out, row * D + d + 1, a.out_dtype, o1);
        }
      }
      if (kV2 && !it.direct && warp == 0 && t == 0) {
        const int64_t w = row * a.num_partitions + it.part;
        a.max_logits[w] = poison ? qnan() : m_run * kLn2;
        a.exp_sums[w] = s_run;
      }
    }
  }
  // one-launch V2: pass 2 by this grid, once every CTA has stored its
  // partials (this CTA's consumer threads meet first: their stores precede
  // the finished count); every block was consumed, so the ring is free
  if (fused) {
    consumer_sync();
    gridred::grid_reduce<D>(a, flags[Lay::kWsOk] != 0, started, red_word,
                            *reinterpret_cast<gridred::UnitScratch*>(ring), &pmap, red_bar, tid,
                            kWaitBudget, false);
  }
  }

  // ---- cluster merge (cs > 1: one item per cluster) -------------------------------
  // Every CTA left its share's (m, s, unnormalised O, poison) at the start of
  // its ring; after a cluster barrier CTA `rank` merges head_dim columns
  // rank * D / cs .. for the item's G heads, with the same log-sum-exp
  // identity as the V2 reduce (weights exp2(m_r - M)), then a second barrier
  // keeps every CTA's shared memory alive until its peers have read it.
  if (cs > 1) {
    sm100::cluster_sync_all();
    if (warp < kConsumerWarps && cid < total_items) {
      const Item it = item_at<BS, Lay::kChunk>(a, nullptr, cid, kV2, rank, cs);
      const int64_t row0 = static_cast<int64_t>(it.b) * Hq + static_cast<int64_t>(it.kvh) * G;
      if (it.any) {
        const int ncol = D / cs;
        const uint32_t mg = sm100::smem_u32(ring);
        for (int e = tid; e < G * ncol; e += kConsumerWarps * 32) {
          const int gh = e / ncol, d = rank * ncol + e % ncol;
          const int64_t row = row0 + gh;
          float M = -INFINITY;
          bool pois = false;
          for (int p = 0; p < cs; ++p) {
            const uint32_t pb = sm100::mapa_shared(mg, static_cast<uint32_t>(p));
            M = fmaxf(M, sm100::ld_shared_cluster_f32(pb + (kMergeM + gh) * 4));
            pois |= sm100::ld_shared_cluster_f32(pb + kMergePoison * 4) != 0.f;
          }
          float S = 0.f, O = 0.f;
          for (int p = 0; p < cs; ++p) {
            const uint32_t pb = sm100::mapa_shared(mg, static_cast<uint32_t>(p));
            const float m = sm100::ld_shared_cluster_f32(pb + (kMergeM + gh) * 4);
            const float w = m == -INFINITY ? 0.f : exp2f(m - M);
            S += w * sm100::ld_shared_cluster_f32(pb + (kMergeS + gh) * 4);
            O += w * sm100::ld_shared_cluster_f32(pb + (kMergeO + gh * D + d) * 4);
          }
          const float res = pois ? qnan() : O / S;
          if (!kV2 || it.direct) {
            store_out(a.out, row * D + d, a.out_dtype, res);
          } else {
            a.tmp_out[(row * a.num_partitions + it.part) * D + d] = res;
            if (rank == 0 && e % ncol == 0) {
              const int64_t w = row * a.num_partitions + it.part;
              a.max_logits[w] = pois ? qnan() : M * kLn2;
              a.exp_sums[w] = S;
            }
          }
        }
      } else if (!kV2 && rank == 0) {  // V1: NaN rows for a bad length, zeros for L = 0
        for (int i = tid; i < G * D; i += kConsumerWarps * 32)
          store_out(a.out, row0 * D + i, a.out_dtype, it.len_ok ? 0.f : qnan());
      }
    }
    sm100::cluster_sync_all();
  }
}

// Kernel attributes, set once per device and instantiation: the dynamic
// shared memory, and clusters of up to 16 CTAs.
template <typename T, int D, int BS, bool V2>
cudaError_t configure_sx(int dev) {
  static std::atomic<bool> configured[128];
  if (configured[dev].load(std::memory_order_acquire)) return cudaSuccess;
  auto kern = pa_sx_kernel<T, D, BS, V2>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       sx::Layout<D, BS>::kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) configured[dev].store(true, std::memory_order_release);
  return e;
}

// Largest cluster size <= want (a power of two) of which at least `need`
// clusters can be resident at once (queried once per device and size).
template <typename T, int D, int BS, bool V2>
int fit_sx_cluster(int dev, int want, int64_t need) {
  static std::atomic<int> resident[128][5];  // [device][log2 size], 0 = not queried yet
  int lg = 0;
  while ((2 << lg) <= want && lg < 4) ++lg;
  for (; lg >= 1; --lg) {
    const int cs = 1 << lg;
    int r = resident[dev][lg].load(std::memory_order_relaxed);
    if (r == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
      cfg.blockDim = dim3(sx::kThreads, 1, 1);
      cfg.dynamicSmemBytes = static_cast<size_t>(sx::Layout<D, BS>::kSmem);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, pa_sx_kernel<T, D, BS, V2>, &cfg) != cudaSuccess) {
        cudaGetLastError();  // a refused size is not an error of the decode call
        n = 0;
      }
      r = n > 0 ? n : -1;
      resident[dev][lg].store(r, std::memory_order_relaxed);
    }
    if (r >= need) return cs;
  }
  return 1;
}

template <typename T, int D, int BS, bool V2>
cudaError_t launch_sx_v(const KernelArgs& a, const CUtensorMap& pm, int64_t items, int sms,
                        cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (cudaError_t e = configure_sx<T, D, BS, V2>(dev)) return e;
  // persistent: at most two CTAs per SM (items dealt out in balanced rounds,
  // or for a compact work list, whose length only the kernel counts, one
  // CTA per slot)
  const int compact = (V2 && a.num_seqs > 1 && a.num_seqs <= sx::kMaxCompactSeqs) ? 1 : 0;
  const int64_t persistent = sms > 0 ? tc_persistent_grid(items, compact != 0, sms) : 0;
  int cs = 1;
  if (persistent == 0 && sms > 0) {
    // Fewer items than SMs: a cluster of cs CTAs (up to 16) shares each item,
    // splitting its 32-token chunks and merging the shares through
    // distributed shared memory, while every CTA keeps at least 8 chunks
    // (256 tokens), below which the merge costs more than the split saves.
    const int range = V2 ? std::min(a.partition_size, a.max_seq_len) : a.max_seq_len;
    int want = 1;
    while (want < 16 && items * want * 2 <= 2LL * sms && want * 2 * 256 <= range) want *= 2;
    if (want > 1 && !a.fused) cs = fit_sx_cluster<T, D, BS, V2>(dev, want, items);
  }
  const int64_t grid = persistent > 0 ? persistent : items * cs;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(sx::kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(sx::Layout<D, BS>::kSmem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cs > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pa_sx_kernel<T, D, BS, V2>, a, pm, items,
                            cs > 1 ? 0 : compact, cs);
}

template <typename T, int D, int BS>
cudaError_t launch_sx_t(const KernelArgs& a, const CUtensorMap& pm, bool v2, cudaStream_t s) {
  const int64_t items =
      static_cast<int64_t>(a.num_seqs) * a.num_kv_heads * (v2 ? a.num_partitions : 1);
  if (items == 0) return cudaSuccess;
  const int sms = sm100_num_sms();
  return v2 ? launch_sx_v<T, D, BS, true>(a, pm, items, sms, s)
            : launch_sx_v<T, D, BS, false>(a, pm, items, sms, s);
}

template <typename T>
cudaError_t launch_sx_dtype(const KernelArgs& a, const CUtensorMap& pm, bool v2, cudaStream_t s) {
  switch (a.head_dim * 100 + a.block_size) {
    case 25616: return launch_sx_t<T, 256, 16>(a, pm, v2, s);
    case 25632: return launch_sx_t<T, 256, 32>(a, pm, v2, s);
    case 12816: return launch_sx_t<T, 128, 16>(a, pm, v2, s);
    case 12832: return launch_sx_t<T, 128, 32>(a, pm, v2, s);
    case 6416: return launch_sx_t<T, 64, 16>(a, pm, v2, s);
    case 6432: return launch_sx_t<T, 64, 32>(a, pm, v2, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
