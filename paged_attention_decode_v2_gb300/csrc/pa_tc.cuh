// pa_tc.cuh -- persistent tensor-core decode kernel for bf16 / f16 caches.
//
// Work items.  A work item is one (sequence, KV head, token range), the
// range being one V2 partition or the whole sequence (V1); all G <= 8 query
// heads of the KV head are served together, so each key/value byte is read
// once per step.  The grid is persistent (two CTAs per SM, or one CTA with a
// deeper ring per item when there are fewer items than SMs); CTA c takes
// items c, c + gridDim.x, ...  For V2 batches of up to 1024 sequences every
// CTA first builds a compact work list (a prefix sum of the sequences'
// partition counts in shared memory), so only existing (sequence, partition,
// KV head) items are enumerated; otherwise the full space is walked in
// partition-major order and empty ranges are skipped.  The shared-memory ring
// keeps streaming from one item into the next (the producer loads the next
// chunk's block ids while the current one streams).
//
// Roles (192 threads, warp-specialised):
//   warp 4      producer: streams q, keys and values into shared memory with
//               TMA (cp.async.bulk.tensor, 128-byte swizzle): keys as one
//               64-element head_dim slice of 128 tokens per 16 KB stage,
//               values as whole KV blocks;
//   warp 5      MMA issuer: tcgen05.mma, accumulators in tensor memory;
//   warps 0-3   softmax + epilogue.
//
// Per chunk of up to 512 tokens of an item:
//   QK^T   S^T[t, h] = sum_d K[t, d] q[h, d]    M = 128 tokens, N = 16, K = d
//   softmax l = S * scale * log2(e); m = chunk max; p = exp2(l - m); sums in
//          f32; p goes to P^T as a 16-bit hi part (columns 0..7) plus the
//          rounded remainder p - hi (columns 8..15), so P.V sees ~16
//          significant bits of p.
//   P.V    O^T[d, n] = sum_t V[t, d] P^T[t, n]  M = 128 (half of head_dim),
//          N = 16, K = 16 tokens; V is the MN-major operand.
// Chunks of one item are combined in registers with the running max and
// rescale (V1 ranges of any length); within a chunk all logits exist before
// the max is taken, so nothing is rescaled per block.
//
// This is Phase 1 of the V2 scheme in commit 4eb83a7e "qwen3_6_scripts",
// paragraph "Implementation (paged_attention_v2_pytorch.py)" (per-partition
// QK^T, softmax and weighted V sum into tmp_output / exp_sums / max_logits),
// with whole tiles staged by bulk asynchronous copies (the SM90+ tier of the
// same page's BlockLoadToShared notes) and the dot products on tensor cores.
//
// Every wait is bounded.  A wait that gives up sets the status word to
// PA_ERR_DEVICE_TIMEOUT and an abort flag that ends every other wait at
// once; issued copies and MMAs are drained (again with a bound) before
// tensor memory is released, and the outputs the CTA writes become NaN.
#pragma once

#include <algorithm>
#include <atomic>
#include <type_traits>

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_grid_reduce.cuh"
#include "pa_sm100.cuh"

namespace pa {

namespace tc {

constexpr int kThreads = 192;
constexpr int kChunk = 512;           // tokens per chunk
constexpr int kTile = 128;            // tokens per QK^T MMA (M)
constexpr int kStageBytes = 16384;    // one ring stage
constexpr int kTmemCols = 128;        // S: 4 tiles x 16 columns, O^T: 2 x 16
constexpr int kOCol = 64;             // first tensor-memory column of O^T
constexpr int kMaxStages = 12;        // barrier slots in the control block
constexpr int kDeepStages = 11;       // ring of the one-CTA-per-SM shape
constexpr int kMaxCompactSeqs = 1024; // V2 batches up to this size use a compact work list
constexpr long long kDefaultWaitBudget = 4000000000LL;  // cycles (about 2 s)
constexpr long long kSelftestWaitBudget = 20000000LL;   // cycles (about 10 ms)

// Two shapes of the same kernel: a 5-stage ring with two CTAs per SM for
// large grids, and an 11-stage (176 KB) ring with one CTA per SM when there
// are fewer work items than SMs, so each CTA keeps more bytes in flight; the
// latter also holds the receive buffer of the cluster combine.
template <int D, int NST>
struct Layout {
  static constexpr int kSlices = D / 64;                  // 64-element head_dim slices
  static constexpr int kHalves = D / 128;                 // 128-row halves of head_dim
  static constexpr int kVTokens = kStageBytes / (D * 2);  // tokens per V stage
  static constexpr int kQOff = NST * kStageBytes;         // 2 q buffers x slices x 1 KB
  static constexpr int kPtOff = kQOff + 2 * kSlices * 1024;
  static constexpr int kCombOff = kPtOff + (kChunk / 16) * 512;
  // cluster combine receive buffer: sums [cs][8][D / cs], statistics [16][20]
  static constexpr int kCombBytes =
      NST == kDeepStages ? ((8 * D + 16 * 20) * 4 + 1023) / 1024 * 1024 : 0;
  static constexpr int kCtrlOff = kCombOff + kCombBytes;
  static constexpr int kPrefixOff = kCtrlOff + 1024;  // only when the work list is compact
  static constexpr int kPrefixBytes = ((kMaxCompactSeqs + 1) * 4 + 63) / 64 * 64;
  static constexpr int kSmem = kPrefixOff + 1024;     // + room to align to 1024
  static constexpr int kSmemCompact = kSmem + kPrefixBytes;
};

struct Ctrl {
  uint64_t full[kMaxStages];   // stage landed (TMA transaction count)
  uint64_t empty[kMaxStages];  // stage consumed (MMA commit)
  uint64_t qfull[2];           // q buffer landed
  uint64_t qempty[2];          // q buffer no longer read by MMAs
  uint64_t s_full;             // chunk logits ready in tensor memory
  uint64_t p_ready;            // P^T written (128 softmax threads arrive)
  uint64_t o_full;             // chunk O^T ready in tensor memory
  uint64_t tail;               // producer-private: a tail value stage landed
  uint64_t drain;              // abort path: all issued MMAs finished
  uint64_t never;              // self-test: nothing ever arrives here
  uint64_t comb_ready;         // cluster: every CTA's partial sums have landed here
  uint64_t red_bar;            // one-launch V2: a reduce unit's tile of partials landed
  int64_t total_items;         // work items to enumerate
  uint32_t tmem;
  int abort;                   // some wait gave up
  int ws_ok;                   // one-launch V2: the workspace carries the init marker
  int red_word[3];             // one-launch V2: thread 0's broadcasts in the reduce
  int scan[8];                 // per-warp totals of the work-list scan
  float red[2][4][8];          // cross-warp max / sum of the softmax warps
};
static_assert(sizeof(Ctrl) <= 1024, "control block");

// One work item, decoded the same way by every role.
struct Item {
  int b, kvh, part;
  int32_t L;       // the sequence's length
  int32_t t0, t1;  // this CTA's token range; empty when t0 >= t1
  bool len_ok;     // 0 <= seq_len <= max_seq_len
  bool any;        // the item's whole range (over all CTAs of a cluster) has tokens
  bool direct;     // V2 with single_direct: the sequence fits this one partition, so
                   // the item's result is the final output (written straight to out)
};

// Coordinates of item k (no global memory read).  With a compact work list
// (prefix[b] = partitions of sequences before b, kept in shared memory) k runs
// over existing (sequence, partition, KV head) triples only; otherwise over
// the full B x Hkv (x NP) space, partition-major, where ranges past a
// sequence's end come out empty.
__device__ __forceinline__ Item item_coords(const KernelArgs& a, const int32_t* prefix, int64_t k,
                                            bool v2) {
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
  it.t0 = v2 ? it.part * a.partition_size : 0;
  it.t1 = it.t0;
  it.L = 0;
  it.len_ok = false;
  it.any = false;
  it.direct = false;
  return it;
}

// The item's token range, given its sequence's length L, and the share of
// it that CTA `rank` of a cluster of `cs` CTAs streams: a balanced run of
// the range's 128-token tiles (the whole range when cs == 1).
__device__ __forceinline__ void item_range(const KernelArgs& a, Item& it, int32_t L, bool v2,
                                           int rank, int cs) {
  it.L = L;
  it.len_ok = seq_len_ok(a, L);
  it.t1 = !it.len_ok ? it.t0 : (v2 ? min(L, it.t0 + a.partition_size) : L);
  it.any = it.t0 < it.t1;
  it.direct = v2 && a.single_direct && it.len_ok && L <= a.partition_size;
  if (cs > 1 && it.any) {
    const int ntiles = (it.t1 - it.t0 + kTile - 1) / kTile;
    const int lo = rank * ntiles / cs, hi = (rank + 1) * ntiles / cs;
    it.t1 = min(it.t1, it.t0 + hi * kTile);
    it.t0 += lo * kTile;  // lo < ntiles, so t0 <= t1 (empty when lo == hi)
  }
}

__device__ __forceinline__ Item item_at(const KernelArgs& a, const int32_t* prefix, int64_t k,
                                        bool v2, int rank, int cs) {
  Item it = item_coords(a, prefix, k, v2);
  item_range(a, it, __ldg(a.seq_lens + it.b), v2, rank, cs);
  return it;
}

// Block-table entry (chunk start c0) / BS + lane of sequence b, for any lane
// whose entry lies inside the table row (so it may be read before the
// sequence's length is known; lanes past the chunk are masked afterwards).
template <int BS>
__device__ __forceinline__ int32_t load_block_id(const KernelArgs& a, int b, int c0, int lane) {
  const int idx = c0 / BS + lane;
  return idx < a.max_blocks_per_seq
             ? __ldg(a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq + idx)
             : 0;
}

__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void fail(Ctrl& c, int32_t* status) {
  c.abort = 1;
  set_status(status, PA_ERR_DEVICE_TIMEOUT);
}


}  // namespace tc

template <typename T, int D, int BS, bool kV2, int NST, int CPS>
__global__ void __launch_bounds__(tc::kThreads, CPS)
    pa_tc_kernel(const KernelArgs a, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap pmap, int64_t grid_items, int compact,
                 int cluster, long long budget) {
  using namespace tc;
  using Lay = Layout<D, NST>;
  static_assert(D == 128 || D == 256, "head_dim");
  static_assert(BS % 16 == 0 && kTile % BS == 0 && Lay::kVTokens % BS == 0, "block size");
  static_assert(NST <= kMaxStages, "ring depth");
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;

  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (sm100::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  uint8_t* qs = smem + Lay::kQOff;
  uint8_t* pt = smem + Lay::kPtOff;
  int32_t* prefix_s = reinterpret_cast<int32_t*>(smem + Lay::kPrefixOff);
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + Lay::kCtrlOff);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.group, Hq = a.num_heads;
  // Clusters of cs CTAs (cs == 1: none) share each work item: cluster cid
  // takes items cid, cid + clusters, ...; CTA `rank` streams its share of the
  // item's tokens and the partial results are merged through distributed
  // shared memory.  Only the one-CTA-per-SM shape is launched in clusters;
  // the persistent two-CTA shape compiles without any of it.
  constexpr bool kClusters = NST == kDeepStages;
  const int cs = kClusters ? cluster : 1;
  const int rank = kClusters ? static_cast<int>(blockIdx.x % cs) : 0;
  const int64_t cid = kClusters ? blockIdx.x / cs : blockIdx.x;
  const int64_t stride = kClusters ? gridDim.x / cs : gridDim.x;

  // The grid is persistent, so every CTA starts at once: let the reduce
  // kernel (a programmatic dependent) be scheduled now; it waits for this
  // grid's results before reading them.
  asm volatile("griddepcontrol.launch_dependents;");

  // Without a compact work list the producer's first item needs nothing the
  // set-up writes: its length and first block ids are loaded now, so the
  // load latency overlaps the set-up below.
  int32_t pre_L = 0, pre_raw = 0;
  const bool pre = warp == 4 && !compact && cid < grid_items;
  if (pre) {
    const Item it0 = item_coords(a, nullptr, cid, kV2);
    pre_L = __ldg(a.seq_lens + it0.b);
    pre_raw = load_block_id<BS>(a, it0.b, it0.t0, lane);
  }

  // ---- set-up -----------------------------------------------------------------
  unsigned long long started = 0;  // thread 0, one-launch V2: the start word as it was
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      sm100::mbar_init(&c.full[s], 1);
      sm100::mbar_init(&c.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      sm100::mbar_init(&c.qfull[s], 1);
      sm100::mbar_init(&c.qempty[s], 1);
    }
    sm100::mbar_init(&c.s_full, 1);
    sm100::mbar_init(&c.p_ready, 128);
    sm100::mbar_init(&c.o_full, 1);
    sm100::mbar_init(&c.tail, 1);
    sm100::mbar_init(&c.drain, 1);
    sm100::mbar_init(&c.never, 1);
    if (kClusters) sm100::mbar_init(&c.comb_ready, 1);
    c.abort = 0;
    // one-launch V2: the counters are usable only in an initialised workspace;
    // the CTA counts itself started (the result is first used at the end)
    if (kV2 && a.fused) {
      sm100::mbar_init(&c.red_bar, 1);
      c.ws_ok = __ldcg(a.status + kMarkerOffset / 4) == kMarker;
      if (c.ws_ok)
        started = gridred::count_started(a);
      else
        set_status(a.status, PA_ERR_WORKSPACE_NOT_INIT);
    }
  }
  if (warp == 5) {
    sm100::tmem_alloc(&c.tmem, kTmemCols);
    sm100::tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    if (kV2 && a.fused) sm100::tma_prefetch_desc(&pmap);
    sm100::tma_prefetch_desc(&kmap);
    sm100::tma_prefetch_desc(&vmap);
    sm100::tma_prefetch_desc(&qmap);
  }
  const int32_t* prefix = nullptr;
  if (compact) {
    // Compact work list: prefix[b] = partitions of the sequences before b.
    // A sequence whose length is outside 0..max_seq_len contributes none
    // (the reduce kernel writes its NaN rows).
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
      if (lane == 31) c.scan[warp] = x;
      __syncthreads();
      int off = 0, round_total = 0;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) {
        off += w < warp ? c.scan[w] : 0;
        round_total += c.scan[w];
      }
      if (b < a.num_seqs) prefix_s[b + 1] = carry + off + x;
      carry += round_total;
      __syncthreads();
    }
    if (tid == 0) {
      prefix_s[0] = 0;
      c.total_items = static_cast<int64_t>(carry) * a.num_kv_heads;
    }
    prefix = prefix_s;
  } else if (tid == 0) {
    c.total_items = grid_items;
  }
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  // peers' barriers must be initialised before any CTA signals them
  if (cs > 1) sm100::cluster_sync_all();
  const uint32_t tmem = c.tmem;
  const int64_t total_items = c.total_items;
  volatile int* abort_flag = &c.abort;

  if (warp == 4) {
    // ========================= producer ===========================================
    const uint64_t stream_once = sm100::l2_evict_first_policy();  // keys and values
    uint64_t keep;                                                // q: default priority
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(keep));
    uint32_t g = 0, qn = 0, tn = 0;  // ring stages / q buffers / tail stages so far
    int tail_pending = -1;           // slot of a tail stage still landing
    bool ok = true;

    // Chunks are visited in order (item k, chunk ci); the block ids of the
    // next chunk are loaded while the current one streams.
    auto next_active = [&](int64_t k, Item& it) -> int64_t {
      for (; k < total_items; k += stride) {
        it = item_at(a, prefix, k, kV2, rank, cs);
        if (it.t0 < it.t1) return k;
      }
      return total_items;
    };
    // TMA row of each lane's block of chunk ci (lanes past the chunk: row 0,
    // never used); a bad id becomes a negative row, which TMA fills with
    // zeros instead of reading memory.
    auto block_rows = [&](const Item& it, int ci, int32_t id, int32_t& y, bool& badl) {
      const int n = min(kChunk, it.t1 - (it.t0 + ci * kChunk));
      const int nblk = (n + BS - 1) / BS;  // <= 32: one block per lane
      badl = lane < nblk && (id < 0 || id >= a.num_blocks);
      y = lane >= nblk ? 0 : badl ? -BS : (id * a.num_kv_heads + it.kvh) * BS;
    };

    // First item: its length and its first chunk's block ids are loaded
    // together (one memory latency before the first copy, not two).
    Item it;
    int64_t k = cid;
    int32_t raw = 0;
    if (k < total_items) {
      it = item_coords(a, prefix, k, kV2);
      const int32_t L = pre ? pre_L : __ldg(a.seq_lens + it.b);
      const int32_t t_spec = it.t0;
      raw = pre ? pre_raw : load_block_id<BS>(a, it.b, t_spec, lane);
      item_range(a, it, L, kV2, rank, cs);
      if (it.t0 < it.t1 && it.t0 != t_spec) raw = load_block_id<BS>(a, it.b, it.t0, lane);
      if (it.t0 >= it.t1) {
        k = next_active(k + stride, it);
        if (k < total_items) raw = load_block_id<BS>(a, it.b, it.t0, lane);
      }
    }
    int ci = 0;
    int32_t y = 0;
    bool badl = false;
    if (k < total_items) block_rows(it, 0, raw, y, badl);
    while (k < total_items && ok) {
      const int nchunks = (it.t1 - it.t0 + kChunk - 1) / kChunk;
      if (__any_sync(0xffffffffu, badl) && lane == 0) set_status(a.status, PA_ERR_BAD_BLOCK_ID);
      if (ci == 0) {
        // q rows of the item's query heads (8 rows; rows past G are ignored)
        const int qb = qn & 1;
        ok = sm100::mbar_wait(&c.qempty[qb], ((qn >> 1) & 1) ^ 1, budget, abort_flag);
        if (!ok) break;
        if (lane == 0) sm100::mbar_arrive_expect_tx(&c.qfull[qb], Lay::kSlices * 1024);
        __syncwarp();
        if (lane < Lay::kSlices)  // one lane per slice
          sm100::tma_load_2d(qs + (qb * Lay::kSlices + lane) * 1024, &qmap, &c.qfull[qb], lane * 64,
                             it.b * Hq + it.kvh * G, keep);
        ++qn;
      }
      const bool tail_fix = (it.t1 % 16) != 0;
      const int c0 = it.t0 + ci * kChunk;
      const int n = min(kChunk, it.t1 - c0);
      const int nt = (n + kTile - 1) / kTile;
      for (int tt = 0; tt < nt && ok; ++tt) {
        const int jb0 = tt * kTile / BS;
        const int jb1 = (min(n, tt * kTile + kTile) + BS - 1) / BS;
        for (int sl = 0; sl < Lay::kSlices; ++sl) {
          const int slot = g % NST;
          ok = sm100::mbar_wait(&c.empty[slot], ((g / NST) & 1) ^ 1, budget, abort_flag);
          if (!ok) break;
          if (lane == 0) sm100::mbar_arrive_expect_tx(&c.full[slot], (jb1 - jb0) * BS * 128);
          __syncwarp();
          // one lane per block: the whole stage is issued by one warp instruction
          const int32_t yj = __shfl_sync(0xffffffffu, y, (jb0 + lane) & 31);
          if (jb0 + lane < jb1)
            sm100::tma_load_2d(ring + slot * kStageBytes + lane * BS * 128, &kmap, &c.full[slot],
                               sl * 64, yj, stream_once);
          ++g;
        }
      }
      // Look ahead while the values stream: the next chunk (of this item, or
      // the next item's first) and its block ids.  The loads are only issued
      // here; their results are first used after the value stages.
      Item it2 = it;
      int64_t k2 = k;
      int ci2 = ci + 1;
      int32_t L2 = 0;
      const bool same_item = ci2 < nchunks;
      if (!same_item) {
        k2 = k + stride;
        ci2 = 0;
        if (k2 < total_items) {
          it2 = item_coords(a, prefix, k2, kV2);
          L2 = __ldg(a.seq_lens + it2.b);
        }
      }
      int32_t raw2 = 0;
      const int32_t t2_spec = it2.t0 + ci2 * kChunk;
      if (k2 < total_items) raw2 = load_block_id<BS>(a, it2.b, t2_spec, lane);
      const int nv = (n + Lay::kVTokens - 1) / Lay::kVTokens;
      for (int v = 0; v < nv && ok; ++v) {
        const int jb0 = v * Lay::kVTokens / BS;
        const int jb1 = (min(n, (v + 1) * Lay::kVTokens) + BS - 1) / BS;
        const int slot = g % NST;
        ok = sm100::mbar_wait(&c.empty[slot], ((g / NST) & 1) ^ 1, budget, abort_flag);
        if (!ok) break;
        // The stage holding the range end, when that end falls inside a
        // 16-token MMA step, lands on the producer's own barrier first: the
        // rows past the end are cleared (P^T is zero there, but 0 * NaN
        // would be NaN) and only then is the stage handed to the MMA warp.
        const bool tail = tail_fix && ci == nchunks - 1 && v == nv - 1;
        uint64_t* land = tail ? &c.tail : &c.full[slot];
        if (lane == 0) sm100::mbar_arrive_expect_tx(land, (jb1 - jb0) * BS * D * 2);
        __syncwarp();
        const int32_t yj = __shfl_sync(0xffffffffu, y, (jb0 + lane) & 31);
        if (jb0 + lane < jb1)
          sm100::tma_load_3d(ring + slot * kStageBytes + lane * BS * D * 2, &vmap, land, 0, yj, 0,
                             stream_once);
        ++g;
        if (tail) {
          tail_pending = slot;
          ok = sm100::mbar_wait(&c.tail, tn & 1, budget, abort_flag);
          if (!ok) break;
          ++tn;
          tail_pending = -1;
          const int r0 = n - v * Lay::kVTokens;  // first row past the end
          const int r1 = (r0 + 15) / 16 * 16;    // end of its 16-token step
          uint8_t* st = ring + slot * kStageBytes;
          const int pieces = (r1 - r0) * Lay::kSlices * 8;  // 16-byte pieces
          for (int i = lane; i < pieces; i += 32) {
            const int line = i / 8, piece = i % 8;
            const int r = r0 + line / Lay::kSlices, sl = line % Lay::kSlices;
            *reinterpret_cast<uint4*>(st + (r / BS) * BS * D * 2 + sl * BS * 128 + (r % BS) * 128 +
                                      piece * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          sm100::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) sm100::mbar_arrive(&c.full[slot]);  // no bytes: the data is there
        }
      }
      if (!same_item && k2 < total_items) {
        item_range(a, it2, L2, kV2, rank, cs);
        if (it2.t0 < it2.t1 && it2.t0 != t2_spec) raw2 = load_block_id<BS>(a, it2.b, it2.t0, lane);
        if (it2.t0 >= it2.t1) {  // an empty item: find the next one with tokens
          k2 = next_active(k2 + stride, it2);
          if (k2 < total_items) raw2 = load_block_id<BS>(a, it2.b, it2.t0, lane);
        }
      }
      k = k2;
      ci = ci2;
      it = it2;
      if (k < total_items) block_rows(it, ci, raw2, y, badl);
    }
    if (!ok) {
      if (lane == 0) fail(c, a.status);
      // Copies already issued must land before the CTA may exit: wait for
      // the newest use of every slot (older uses completed before it began).
      for (uint32_t gg = g > NST ? g - NST : 0; gg < g; ++gg)
        if (static_cast<int>(gg % NST) != tail_pending)
          sm100::mbar_wait(&c.full[gg % NST], (gg / NST) & 1, budget, nullptr);
      if (tail_pending >= 0) sm100::mbar_wait(&c.tail, tn & 1, budget, nullptr);
      for (uint32_t qq = qn > 2 ? qn - 2 : 0; qq < qn; ++qq)
        sm100::mbar_wait(&c.qfull[qq & 1], (qq >> 1) & 1, budget, nullptr);
    }
  } else if (warp == 5) {
    // ========================= MMA issuer =========================================
    // The whole warp runs the loop (waits, descriptors) in convergent code and
    // one elected lane issues each MMA and commit; every branch below depends
    // on warp-uniform values only (a wait's result is agreed with __all_sync).
    {
      constexpr unsigned kAll = 0xffffffffu;
      constexpr uint32_t id_qk = sm100::idesc_f16(kBf16, false, false, 128, 16);
      constexpr uint32_t id_pv = sm100::idesc_f16(kBf16, true, false, 128, 16);
      const uint32_t q_base = sm100::smem_u32(qs);
      const uint32_t pt_base = sm100::smem_u32(pt);
      const uint32_t ring_base = sm100::smem_u32(ring);
      uint32_t g = 0, qn = 0, cc = 0;
      bool ok = true;
      // diagnostic: wait for an event that never happens, so the bounded
      // wait runs out and the abort path is exercised
      if (a.selftest_stall) ok = __all_sync(kAll, sm100::mbar_wait(&c.never, 0, budget, abort_flag));
      for (int64_t k = cid; k < total_items && ok; k += stride) {
        const Item it = item_at(a, prefix, k, kV2, rank, cs);
        if (it.t0 >= it.t1) continue;
        const int qb = qn & 1;
        ok = __all_sync(kAll, sm100::mbar_wait(&c.qfull[qb], (qn >> 1) & 1, budget, abort_flag));
        if (!ok) break;
        ++qn;
        const uint32_t qbuf = q_base + qb * Lay::kSlices * 1024;
        const int nchunks = (it.t1 - it.t0 + kChunk - 1) / kChunk;
        for (int ci = 0; ci < nchunks && ok; ++ci, ++cc) {
          const int c0 = it.t0 + ci * kChunk;
          const int n = min(kChunk, it.t1 - c0);
          const int nt = (n + kTile - 1) / kTile;
          for (int tt = 0; tt < nt && ok; ++tt) {
            for (int sl = 0; sl < Lay::kSlices; ++sl) {
              const int slot = g % NST;
              ok = __all_sync(kAll, sm100::mbar_wait(&c.full[slot], (g / NST) & 1, budget, abort_flag));
              if (!ok) break;
              sm100::tc_fence_after();
              const uint32_t st = ring_base + slot * kStageBytes;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = sm100::smem_desc(st + kk * 32, 16, 1024, sm100::kSw128);
                const uint64_t bd =
                    sm100::smem_desc(qbuf + sl * 1024 + kk * 32, 16, 1024, sm100::kSw128);
                sm100::mma_f16_elect(tmem + tt * 16, ad, bd, id_qk, (sl | kk) != 0);
              }
              sm100::mma_commit_elect(&c.empty[slot]);
              ++g;
            }
          }
          if (!ok) break;
          if (ci == nchunks - 1) sm100::mma_commit_elect(&c.qempty[qb]);
          sm100::mma_commit_elect(&c.s_full);
          ok = __all_sync(kAll, sm100::mbar_wait(&c.p_ready, cc & 1, budget, abort_flag));
          if (!ok) break;
          sm100::tc_fence_after();
          const int nv = (n + Lay::kVTokens - 1) / Lay::kVTokens;
          bool first = true;
          for (int v = 0; v < nv; ++v) {
            const int slot = g % NST;
            ok = __all_sync(kAll, sm100::mbar_wait(&c.full[slot], (g / NST) & 1, budget, abort_flag));
            if (!ok) break;
            sm100::tc_fence_after();
            const uint32_t st = ring_base + slot * kStageBytes;
            const int toks = min(Lay::kVTokens, n - v * Lay::kVTokens);
            for (int r = 0; r < toks; r += 16) {
              const int jb = r / BS, s0 = r % BS;
              const uint64_t bd = sm100::smem_desc(pt_base + ((v * Lay::kVTokens + r) / 16) * 512,
                                                   256, 128, sm100::kSwNone);
#pragma unroll
              for (int j = 0; j < Lay::kHalves; ++j) {
                const uint64_t ad =
                    sm100::smem_desc(st + jb * BS * D * 2 + 2 * j * BS * 128 + s0 * 128, BS * 128,
                                     1024, sm100::kSw128);
                sm100::mma_f16_elect(tmem + kOCol + 16 * j, ad, bd, id_pv, !first);
              }
              first = false;
            }
            sm100::mma_commit_elect(&c.empty[slot]);
            ++g;
          }
          if (!ok) break;
          sm100::mma_commit_elect(&c.o_full);
        }
      }
      if (!ok) {
        if (lane == 0) fail(c, a.status);
        // no MMA may still be running when tensor memory is released
        sm100::mma_commit_elect(&c.drain);
        sm100::mbar_wait(&c.drain, 0, budget, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ========================= softmax + epilogue (warps 0-3) =====================
    // Every softmax thread runs the same iterations and barriers whatever
    // happens; a failed wait only marks the abort, which ends later waits.
    const int r = tid;  // tensor-memory lane: token of a tile, or head_dim row
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = a.scale_log2;
    // Cluster combine of the cluster's item (the host launches one cluster
    // per item, so each CTA combines once and no buffer is reused).  The CTA
    // that merges head_dim elements [r * D / cs, (r + 1) * D / cs) is CTA r:
    // every CTA pushes its unnormalised P.V sums for those elements, and its
    // running max (log2 units), running sum and poison flag, into CTA r's
    // combine buffer with remote stores counted on CTA r's mbarrier; CTA r
    // then merges them with the same log-sum-exp identity as the V2 reduce
    // and writes the output.
    auto combine = [&](const float (&acc)[Lay::kHalves][8], const float (&m_run)[8],
                       const float (&s_run)[8], bool poison, const Item& it, int64_t row0,
                       uint64_t keep_l2, uint32_t ic) {
      const int dn = D / cs;  // head_dim elements each CTA merges
      // receive side: its own buffer, since a peer may push while this CTA's
      // last P.V still reads its P^T
      float* recv = reinterpret_cast<float*>(smem + Lay::kCombOff);  // [cs][8][dn] sums
      float* rst = recv + 8 * D;                                     // [cs][20] statistics
      const uint32_t bar_s = sm100::smem_u32(&c.comb_ready);
      if (tid == 0)
        sm100::mbar_arrive_expect_tx(&c.comb_ready,
                                     static_cast<uint32_t>(cs * (G * dn + 20) * 4));
      // send side: stage the sums in the P^T buffer (idle: this CTA's last
      // P.V has completed) and push them as 16-byte pieces
      float* xo = reinterpret_cast<float*>(pt);  // [8][D]
#pragma unroll
      for (int j = 0; j < Lay::kHalves; ++j)
#pragma unroll
        for (int h = 0; h < 8; ++h)
          if (h < G) xo[h * D + j * 128 + tid] = acc[j][h];
      softmax_sync();
      for (int u = tid; u < G * (D / 4); u += 128) {
        const int h = u / (D / 4), d = (u % (D / 4)) * 4;
        const uint32_t owner = static_cast<uint32_t>(d / dn);
        const float4 v = *reinterpret_cast<const float4*>(xo + h * D + d);
        sm100::st_async_v4(
            sm100::mapa_shared(sm100::smem_u32(recv + (rank * 8 + h) * dn + d % dn), owner), v,
            sm100::mapa_shared(bar_s, owner));
      }
      if (tid < cs) {  // statistics: max[8], sum[8], poison, padding
        const uint32_t dst = sm100::mapa_shared(sm100::smem_u32(rst + rank * 20), tid);
        const uint32_t bar = sm100::mapa_shared(bar_s, tid);
        sm100::st_async_v4(dst, make_float4(m_run[0], m_run[1], m_run[2], m_run[3]), bar);
        sm100::st_async_v4(dst + 16, make_float4(m_run[4], m_run[5], m_run[6], m_run[7]), bar);
        sm100::st_async_v4(dst + 32, make_float4(s_run[0], s_run[1], s_run[2], s_run[3]), bar);
        sm100::st_async_v4(dst + 48, make_float4(s_run[4], s_run[5], s_run[6], s_run[7]), bar);
        sm100::st_async_v4(dst + 64, make_float4(poison ? 1.f : 0.f, 0.f, 0.f, 0.f), bar);
      }
      const bool ready = sm100::mbar_wait_cluster(&c.comb_ready, ic & 1, budget, abort_flag);
      if (!ready) fail(c, a.status);
      // merge: each thread derives its head's weights from the statistics
      bool pz = !ready;
      for (int q = 0; q < cs; ++q) pz |= rst[q * 20 + 16] != 0.f;
      for (int i = tid; i < G * dn; i += 128) {
        const int h = i / dn, dl = i % dn, d = rank * dn + dl;
        float M = -INFINITY;
        for (int q = 0; q < cs; ++q) M = fmaxf(M, rst[q * 20 + h]);
        float S = 0.f, O = 0.f;
        for (int q = 0; q < cs; ++q) {
          const float mq = rst[q * 20 + h];
          const float f = mq == -INFINITY ? 0.f : exp2f(mq - M);
          S = fmaf(rst[q * 20 + 8 + h], f, S);
          O = fmaf(recv[(q * 8 + h) * dn + dl], f, O);
        }
        const float o = pz ? qnan() : O / S;
        if (kV2 && !it.direct) {
          sm100::st_f32_policy(a.tmp_out + ((row0 + h) * a.num_partitions + it.part) * D + d, o,
                               keep_l2);
          if (rank == 0 && dl == 0) {
            const int64_t w = (row0 + h) * a.num_partitions + it.part;
            sm100::st_f32_policy(a.max_logits + w, pz ? qnan() : M * kLn2, keep_l2);
            sm100::st_f32_policy(a.exp_sums + w, S, keep_l2);
          }
        } else {
          store_out(a.out, (row0 + h) * D + d, a.out_dtype, o);
        }
      }
    };
    // One-launch V2: run the end-of-kernel reduce once now, dry (no side
    // effects, scratch in the still unused P^T buffer), while the first keys
    // land, so its code is in the instruction cache when the reduce runs.
    static_assert(gridred::kDryBytes <= (kChunk / 16) * 512, "dry run within the P^T buffer");
    if (kV2 && !kClusters && a.fused && c.ws_ok) {
      uint32_t dry_phase = 0;
      gridred::grid_reduce<D>(a, true, started, c.red_word,
                              *reinterpret_cast<gridred::UnitScratch*>(pt), &pmap, &c.red_bar,
                              tid, budget, true);
      gridred::reduce_unit<D>(a, &pmap, &c.red_bar, dry_phase, 0, 0,
                              *reinterpret_cast<gridred::UnitScratch*>(pt), tid, false, budget,
                              true);
    }
    uint32_t cc = 0, ic = 0;  // chunks / cluster combines so far
    for (int64_t k = cid; k < total_items; k += stride) {
      const Item it = item_at(a, prefix, k, kV2, rank, cs);
      const int64_t row0 = static_cast<int64_t>(it.b) * Hq + it.kvh * G;
      if (!it.any) {  // nothing to attend to in the whole item
        if (rank == 0) {
          if (!it.len_ok && it.part == 0 && it.kvh == 0 && tid == 0)
            set_status(a.status, PA_ERR_BAD_SEQ_LEN);
          if (!kV2) {  // V1 row of a sequence with nothing to attend to
            const float v = it.len_ok ? 0.f : qnan();
            for (int i = tid; i < G * D; i += 128) store_out(a.out, row0 * D + i, a.out_dtype, v);
          }
        }
        continue;
      }
      const int32_t* bt = a.block_tables + static_cast<int64_t>(it.b) * a.max_blocks_per_seq;
      float m_run[8], s_run[8], acc[Lay::kHalves][8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        m_run[h] = -INFINITY;
        s_run[h] = 0.f;
#pragma unroll
        for (int j = 0; j < Lay::kHalves; ++j) acc[j][h] = 0.f;
      }
      bool bad = false;
      const int nchunks = (it.t1 - it.t0 + kChunk - 1) / kChunk;
      for (int ci = 0; ci < nchunks; ++ci, ++cc) {
        const int c0 = it.t0 + ci * kChunk;
        const int n = min(kChunk, it.t1 - c0);
        const int nt = (n + kTile - 1) / kTile;
        const int n16 = (n + 15) / 16 * 16;
        {  // block ids of the chunk: any outside the pool poisons the item
          const int nblk = (n + BS - 1) / BS;
          bool bl = false;
          if (lane < nblk) {
            const int32_t id = __ldg(bt + c0 / BS + lane);
            bl = id < 0 || id >= a.num_blocks;
          }
          bad |= __any_sync(0xffffffffu, bl);
        }
        if (!sm100::mbar_wait(&c.s_full, cc & 1, budget, abort_flag)) fail(c, a.status);
        sm100::tc_fence_after();
        __syncwarp();
        float mx[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) mx[h] = -INFINITY;
        for (int tt = 0; tt < nt; ++tt) {
          float s[16];
          sm100::tmem_ld16(tmem + lane_base + tt * 16, s);
          sm100::tmem_wait_ld();
          if (tt * kTile + r < n) {
#pragma unroll
            for (int h = 0; h < 8; ++h)
              if (h < G) mx[h] = fmaxf(mx[h], s[h] * sl2);
          }
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) {
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1)
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], o));
          if (lane == 0) c.red[0][warp][h] = mx[h];
        }
        softmax_sync();
        float mc[8];
#pragma unroll
        for (int h = 0; h < 8; ++h)
          mc[h] = fmaxf(fmaxf(c.red[0][0][h], c.red[0][1][h]), fmaxf(c.red[0][2][h], c.red[0][3][h]));
        float sum[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) sum[h] = 0.f;
        for (int tt = 0; tt < nt; ++tt) {
          float s[16];
          sm100::tmem_ld16(tmem + lane_base + tt * 16, s);
          sm100::tmem_wait_ld();
          const int tok = tt * kTile + r;
          if (tok < n16) {
            const bool valid = tok < n;
            // P^T element (tok, col): 16-token step, 8-token core, column
            // group col / 8, column col % 8, token tok % 8 (no-swizzle
            // K-major core matrices of 8 x 16 bytes)
            uint8_t* dst = pt + (tok / 16) * 512 + ((tok % 16) / 8) * 256 + (tok % 8) * 2;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              float p = 0.f;
              if (valid && h < G) p = exp2f(s[h] * sl2 - mc[h]);
              sum[h] += p;
              const T hi = round16(p, static_cast<T*>(nullptr));
              const T lo = round16(p - to_float(hi), static_cast<T*>(nullptr));
              *reinterpret_cast<uint16_t*>(dst + h * 16) = bits16(hi);
              *reinterpret_cast<uint16_t*>(dst + 128 + h * 16) = bits16(lo);
            }
          }
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) {
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], o);
          if (lane == 0) c.red[1][warp][h] = sum[h];
        }
        sm100::fence_proxy_async_smem();
        sm100::tc_fence_before();
        sm100::mbar_arrive(&c.p_ready);
        softmax_sync();
        float f_old[8], f_new[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float sc = (c.red[1][0][h] + c.red[1][1][h]) + (c.red[1][2][h] + c.red[1][3][h]);
          const float m_new = fmaxf(m_run[h], mc[h]);
          f_old[h] = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - m_new);
          f_new[h] = mc[h] == -INFINITY ? 0.f : exp2f(mc[h] - m_new);
          s_run[h] = s_run[h] * f_old[h] + sc * f_new[h];
          m_run[h] = m_new;
        }
        if (!sm100::mbar_wait(&c.o_full, cc & 1, budget, abort_flag)) fail(c, a.status);
        sm100::tc_fence_after();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < Lay::kHalves; ++j) {
          float o[16];
          sm100::tmem_ld16(tmem + lane_base + kOCol + 16 * j, o);
          sm100::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 8; ++h)
            acc[j][h] = acc[j][h] * f_old[h] + (o[h] + o[8 + h]) * f_new[h];
        }
        sm100::tc_fence_before();
      }
      // ---- epilogue of the item ------------------------------------------------
      // partials are read back by the reduce right after this kernel: keep
      // them in L2 (the key / value stream is marked evict-first)
      const uint64_t keep_l2 = sm100::l2_evict_last_policy();
      const bool poison = bad || *abort_flag != 0;
      if (cs > 1) {
        combine(acc, m_run, s_run, poison, it, row0, keep_l2, ic);
        ++ic;
        continue;
      }
#pragma unroll
      for (int j = 0; j < Lay::kHalves; ++j) {
        const int d = j * 128 + tid;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          if (h >= G) break;
          const float o = poison ? qnan() : acc[j][h] / s_run[h];
          if (kV2 && !it.direct)
            sm100::st_f32_policy(a.tmp_out + ((row0 + h) * a.num_partitions + it.part) * D + d, o,
                               keep_l2);
          else
            store_out(a.out, (row0 + h) * D + d, a.out_dtype, o);
        }
      }
      if (kV2 && !it.direct && tid < G) {
        const int64_t w = (row0 + tid) * a.num_partitions + it.part;
        float m = m_run[0], s = s_run[0];
#pragma unroll
        for (int h = 1; h < 8; ++h)
          if (h == tid) {
            m = m_run[h];
            s = s_run[h];
          }
        sm100::st_f32_policy(a.max_logits + w, poison ? qnan() : m * kLn2, keep_l2);
        sm100::st_f32_policy(a.exp_sums + w, s, keep_l2);
      }
    }
  }

  // ---- teardown -------------------------------------------------------------------
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  if (warp == 5) sm100::tmem_dealloc(tmem, kTmemCols);
  // one-launch V2 (persistent shape only): pass 2 by this grid, once every
  // CTA has stored its partials; the ring is free scratch now
  static_assert(sizeof(gridred::UnitScratch) <= NST * kStageBytes, "reduce scratch in the ring");
  static_assert(alignof(gridred::UnitScratch) <= 1024, "the ring starts 1024-byte aligned");
  if (kV2 && !kClusters && a.fused && warp < 4)
    gridred::grid_reduce<D>(a, c.ws_ok != 0, started, c.red_word,
                            *reinterpret_cast<gridred::UnitScratch*>(ring), &pmap, &c.red_bar, tid,
                            budget, false);
  // no CTA leaves while a peer may still read its shared memory
  if (cs > 1) sm100::cluster_sync_all();
}

// Kernel attributes, set once per device: the dynamic shared memory, and for
// the one-CTA-per-SM variant clusters of up to 16 CTAs.
template <typename T, int D, int BS, bool V2, int NST, int CPS>
cudaError_t configure_tc(int dev) {
  // set once per device; concurrent first calls set the same attributes
  static std::atomic<bool> configured[128];
  if (configured[dev].load(std::memory_order_acquire)) return cudaSuccess;
  auto kern = pa_tc_kernel<T, D, BS, V2, NST, CPS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       tc::Layout<D, NST>::kSmemCompact);
  if (e == cudaSuccess && NST == tc::kDeepStages)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) configured[dev].store(true, std::memory_order_release);
  return e;
}

template <typename T, int D, int BS, bool V2, int NST, int CPS>
cudaError_t launch_tc_variant(const KernelArgs& a, const CUtensorMap& km, const CUtensorMap& vm,
                              const CUtensorMap& qm, const CUtensorMap& pm, int64_t items,
                              unsigned grid, int compact, int cs, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  auto kern = pa_tc_kernel<T, D, BS, V2, NST, CPS>;
  using Lay = tc::Layout<D, NST>;
  // the compact work list's prefix table only takes shared memory when used,
  // which leaves room on each SM for the reduce kernel's waiting CTAs
  const int smem = compact ? Lay::kSmemCompact : Lay::kSmem;
  if (cudaError_t e = configure_tc<T, D, BS, V2, NST, CPS>(dev)) return e;
  const long long budget = a.selftest_stall ? tc::kSelftestWaitBudget : tc::kDefaultWaitBudget;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(tc::kThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cs > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, km, vm, qm, pm, items, compact, cs, budget);
}

// Largest cluster size <= want (a power of two) of which at least `need`
// clusters of the one-CTA-per-SM variant can be resident at once.  The
// resident-cluster counts are queried once per device and size.
template <typename T, int D, int BS, bool V2>
int fit_cluster(int want, int64_t need) {
  // [device][log2 size], 0 = not queried yet; concurrent first calls store the same count
  static std::atomic<int> resident[128][5];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 1;
  if (configure_tc<T, D, BS, V2, tc::kDeepStages, 1>(dev) != cudaSuccess) return 1;
  auto kern = pa_tc_kernel<T, D, BS, V2, tc::kDeepStages, 1>;
  int lg = 0;
  while ((2 << lg) <= want && lg < 4) ++lg;  // log2 of the largest power of two <= want
  for (; lg >= 1; --lg) {
    const int cs = 1 << lg;
    int r = resident[dev][lg].load(std::memory_order_relaxed);
    if (r == 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
      cfg.blockDim = dim3(tc::kThreads, 1, 1);
      cfg.dynamicSmemBytes = static_cast<size_t>(tc::Layout<D, tc::kDeepStages>::kSmemCompact);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
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

template <typename T, int D, int BS>
cudaError_t launch_tc_t(const KernelArgs& a, const CUtensorMap& km, const CUtensorMap& vm,
                        const CUtensorMap& qm, const CUtensorMap& pm, bool v2, int num_sms,
                        cudaStream_t s) {
  // upper bound of the work items: every (sequence, KV head[, partition])
  const int64_t items = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads *
                        (v2 ? a.num_partitions : 1);
  if (items == 0) return cudaSuccess;
  const int compact = (v2 && a.num_seqs > 1 && a.num_seqs <= tc::kMaxCompactSeqs) ? 1 : 0;
  const int64_t persistent = tc_persistent_grid(items, compact != 0, num_sms);
  if (persistent == 0) {
    // Few items: one deep-ring CTA per SM, and when at most half the SMs
    // would be busy, each item is shared by a cluster of cs CTAs (up to 16)
    // that split its 128-token tiles and merge their partial results -- as
    // long as every CTA keeps at least four tiles (512 tokens), below which
    // the merge costs more than the split saves.
    const int range = v2 ? std::min(a.partition_size, a.max_seq_len) : a.max_seq_len;
    const int tiles = (range + tc::kTile - 1) / tc::kTile;
    int want = 1;
    while (want < 16 && items * want * 2 <= num_sms && want * 2 * 4 <= tiles) want *= 2;
    const int cs = want > 1 ? (v2 ? fit_cluster<T, D, BS, true>(want, items)
                                  : fit_cluster<T, D, BS, false>(want, items))
                            : 1;
    const unsigned grid = static_cast<unsigned>(items * cs);
    return v2 ? launch_tc_variant<T, D, BS, true, tc::kDeepStages, 1>(a, km, vm, qm, pm, items, grid, compact, cs, s)
              : launch_tc_variant<T, D, BS, false, tc::kDeepStages, 1>(a, km, vm, qm, pm, items, grid, compact, cs,
                                                          s);
  }
  // Persistent grid: at most two CTAs per SM, every CTA doing the same number
  // of rounds when the items are all the same size (tc_persistent_grid).
  const unsigned grid = static_cast<unsigned>(persistent);
  return v2 ? launch_tc_variant<T, D, BS, true, 5, 2>(a, km, vm, qm, pm, items, grid, compact, 1, s)
            : launch_tc_variant<T, D, BS, false, 5, 2>(a, km, vm, qm, pm, items, grid, compact, 1, s);
}

template <typename T>
cudaError_t launch_tc_dtype(const KernelArgs& a, const CUtensorMap& km, const CUtensorMap& vm,
                            const CUtensorMap& qm, const CUtensorMap& pm, bool v2, int num_sms,
                            cudaStream_t s) {
  if (a.head_dim == 256 && a.block_size == 16)
    return launch_tc_t<T, 256, 16>(a, km, vm, qm, pm, v2, num_sms, s);
  if (a.head_dim == 256 && a.block_size == 32)
    return launch_tc_t<T, 256, 32>(a, km, vm, qm, pm, v2, num_sms, s);
  if (a.head_dim == 128 && a.block_size == 16)
    return launch_tc_t<T, 128, 16>(a, km, vm, qm, pm, v2, num_sms, s);
  if (a.head_dim == 128 && a.block_size == 32)
    return launch_tc_t<T, 128, 32>(a, km, vm, qm, pm, v2, num_sms, s);
  if (a.head_dim == 128 && a.block_size == 64)
    return launch_tc_t<T, 128, 64>(a, km, vm, qm, pm, v2, num_sms, s);
  return cudaErrorInvalidValue;
}

}  // namespace pa
