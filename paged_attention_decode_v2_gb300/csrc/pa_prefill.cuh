// pa_prefill.cuh -- paged prefix prefill on the tensor cores (tcgen05).
//
// A chunk of n_b new tokens of sequence b attends to the sequence's C_b
// cached tokens (read from the paged cache through the block table) and,
// causally, to the chunk itself: commit 1a4e1005 "paged_attn.py", opening
// paragraph (Flash-Attention-style online softmax over key tiles), and
// commit 4eb83a7e "qwen3_6_scripts", paragraphs on the prefix attention's
// pre-allocated m_blk / m_new / corr buffers (a tile loop over the context,
// then one over the chunk), "Complete rewrite of qwen3_6_scripts/
// paged_attn.py" item 1 (the context comes from the cache) and "Prefill
// (flash_attn_func)" (causal=True).
//
// Work unit: (sequence, query head, 128-query tile of the chunk).  A
// persistent grid of one CTA per SM walks the units longest first: last
// query tile first, or, for batches whose contexts differ, by cost (key
// tiles) -- see Walk.  Per unit the key tiles
// (128 keys each) are the context tiles, then the chunk's tiles up to the
// diagonal one; each tile runs
//   QK^T  S[q, k] = sum_d Q[q, d] K[k, d]     M = 128 queries, N = 128 keys,
//         into one of two tensor-memory buffers (the next tile's QK^T runs
//         while the softmax warps work on this one);
//   softmax (two threads per query row): tile max over the visible keys, the
//         running reference max m moves (and the running sum and the output
//         are rescaled by corr = 2^(m_old - m_new)) only when the tile max
//         exceeds it by more than 2^8, so p = 2^(s - m) <= 256; p is rounded
//         to 16 bits for the MMA and the running sum adds the rounded
//         values, so the result is an exact weighted mean of the values with
//         weights perturbed by at most one rounding each; P is written to
//         tensor memory over the tile's logits;
//   P.V   O[q, d] += sum_k P[q, k] V[k, d]    M = 128, N = head_dim, K = keys,
//         A = P from tensor memory, B = V from shared memory (MN-major),
//         accumulated in tensor memory.
// Roles: warps 9 .. 8 + kProducers stream q, keys and values with TMA into a
// ring of 16 KB stages (each issues every kProducers-th stage: a context key
// stage takes one copy per cache block, and one warp issues copies at a
// limited rate); warp 8 issues the MMAs; warps 0-7 run the softmax and the
// epilogue, two threads per query row (warps w and w + 4 read the same
// tensor-memory lanes): one takes keys 0-63 of each tile and the first half
// of head_dim, the other keys 64-127 and the second half; they agree on the
// row's reference max through shared memory once per tile.  Every wait is bounded; a wait that
// gives up makes the CTA's outputs NaN.
#pragma once

#include <algorithm>
#include <atomic>
#include <type_traits>

#include <cuda.h>

#include "pa_device.cuh"
#include "pa_sm100.cuh"

namespace pa {

namespace pf {

constexpr int kProducers = 3;        // producer warps (each issues every kProducers-th stage)
constexpr int kThreads = 288 + 32 * kProducers;
constexpr int kSoftmaxThreads = 256; // warps 0-7
constexpr int kMmaWarp = 8;         // warps 9 .. 8 + kProducers are the producers
constexpr int kTile = 128;          // queries per unit and keys per key tile
constexpr int kStage = 16384;       // one ring stage
constexpr int kMaxStages = 12;      // barrier slots in the control block
constexpr int kTmemCols = 512;      // S0 | S1 | O
constexpr int kS1Col = 128;         // second logits buffer
constexpr int kOCol = 256;          // output accumulator (head_dim columns)
constexpr float kRescaleLog2 = 8.f; // move the reference max past 2^8 growth only
constexpr long long kWaitBudget = 4000000000LL;    // cycles (about 2 s)
constexpr long long kSelftestBudget = 20000000LL;  // cycles (about 10 ms)
constexpr int kSmemLimit = 227 * 1024;

// Shared memory: q (head_dim / 64 slices of [128 rows][128 B]), the ring,
// the control block.  Every operand tile starts on a 1024-byte boundary
// (128-byte swizzle atoms).  P lives in tensor memory, not here: the P.V MMA
// reads it as its A operand where the tile's logits were (below), which
// keeps its 64 KB of writes and reads per tile off the shared-memory
// bandwidth that the MMAs' operand reads and the TMA copies share.
template <int D>
struct Layout {
  static constexpr int kSlices = D / 64;
  static constexpr int kVTokens = kStage / (D * 2);  // keys per value stage
  static constexpr int kRingOff = kSlices * kStage;
  static constexpr int kStages =
      std::min(kMaxStages, (kSmemLimit - kRingOff - 2048) / kStage);
  static constexpr int kCtrlOff = kRingOff + kStages * kStage;
  static constexpr int kSmem = kCtrlOff + 1024 + 1024;  // + room to align to 1024
  static_assert(kSmem <= kSmemLimit, "shared memory");
  static_assert(kStages >= 4, "ring depth");
};

struct Ctrl {
  uint64_t full[kMaxStages];   // stage landed
  uint64_t empty[kMaxStages];  // stage consumed by its MMAs
  uint64_t qfull;              // q tile landed
  uint64_t qempty;             // q tile no longer read
  uint64_t s_full[2];          // a tile's logits ready (per buffer)
  uint64_t p_ready;            // P written (the 256 softmax threads arrive)
  uint64_t o_done[2];          // P.V of a tile completed (by tile parity)
  uint64_t tail[kProducers];   // producer-private: a tail value stage landed
  uint64_t drain;              // abort path: all issued MMAs finished
  uint64_t never;              // self-test: nothing ever arrives here
  uint32_t tmem;
  int abort;
  float xrow[kTile];           // per query row: one half's value for the other half
};
static_assert(sizeof(Ctrl) <= 1024, "control block");

// One work unit, decoded the same way by every role.
struct Unit {
  int b, h, qt;
  int32_t s0;      // first row of the sequence's chunk
  int32_t n;       // chunk tokens
  int32_t C;       // context tokens (0 when invalid)
  bool run;        // the unit exists and its sequence's rows are trusted
  bool poison;     // the context length is invalid: rows become NaN
  int nctx;        // context key tiles
  int ntiles;      // context tiles + chunk tiles up to the diagonal
};

// Unit (sequence b, query head h, query tile qt).
__device__ __forceinline__ Unit unit_of(const PrefillArgs& a, int b, int h, int qt) {
  Unit u;
  u.qt = qt;
  u.b = b;
  u.h = h;
  u.s0 = __ldg(a.query_start + u.b);
  const int32_t s1 = __ldg(a.query_start + u.b + 1);
  u.n = s1 - u.s0;
  const int32_t C = __ldg(a.ctx_lens + u.b);
  const bool seq_ok = u.s0 >= 0 && u.n >= 0 && u.n <= a.max_query_len && s1 <= a.total_tokens;
  u.run = seq_ok && u.qt * kTile < u.n;
  const bool ctx_ok = C >= 0 && C <= a.max_ctx_len &&
                      static_cast<int64_t>(C) <= static_cast<int64_t>(a.max_blocks_per_seq) *
                                                     a.block_size;
  u.poison = !ctx_ok;
  u.C = ctx_ok ? C : 0;
  u.nctx = (u.C + kTile - 1) / kTile;
  u.ntiles = u.nctx + u.qt + 1;
  return u;
}

// The units one CTA processes, in order; every role walks the same sequence.
//  * default: index k = blockIdx.x, + gridDim.x, ... over (query tile
//    descending, sequence, head) -- last query tiles first, which is
//    longest first when every sequence has the same context;
//  * cost order (a.cost_levels > 0, batches of uneven contexts): the units
//    sorted by cost -- key tiles, nctx + qt + 1 -- from the highest level
//    down, then by sequence and head, and this CTA takes every gridDim.x-th
//    one, so the longest units start first (a longest-first static
//    schedule).  Each role scans the (level, sequence) pairs in order;
//    the host enables it only when there are few of them.
struct Walk {
  int64_t k = 0;   // default order: next index
  int c = 0;       // cost order: current level, sequence, its query tile
  int b = 0, qt = 0;
  int h = 0;       //   next head of the current pair for this CTA
  int64_t n0 = 0;  //   units of the pairs before the current one
  bool pair = false;
};

__device__ __forceinline__ Walk walk_begin(const PrefillArgs& a) {
  Walk w;
  w.k = blockIdx.x;
  w.c = a.cost_levels;
  w.b = -1;
  return w;
}

// kCost: the cost order (a.cost_levels > 0); a template parameter so that
// the default walk compiles to the plain index stride.
template <bool kCost>
__device__ __forceinline__ bool walk_next(const PrefillArgs& a, Walk& w, Unit& u) {
  if constexpr (!kCost) {
    const int64_t per = static_cast<int64_t>(a.num_seqs) * a.num_heads;
    const int64_t units = per * a.qtiles;
    while (w.k < units) {
      const int64_t k = w.k;
      w.k += gridDim.x;
      const int64_t rem = k % per;
      u = unit_of(a, static_cast<int>(rem / a.num_heads), static_cast<int>(rem % a.num_heads),
                  a.qtiles - 1 - static_cast<int>(k / per));
      if (u.run) return true;
    }
    return false;
  } else {
    while (true) {
      if (w.pair && w.h < a.num_heads) {
        u = unit_of(a, w.b, w.h, w.qt);
        w.h += gridDim.x;
        return true;
      }
      if (w.pair) w.n0 += a.num_heads;
      if (++w.b >= a.num_seqs) {
        w.b = 0;
        if (--w.c < 1) return false;
      }
      // does sequence b have a unit of cost c, i.e. query tile c - 1 - nctx?
      const Unit s = unit_of(a, w.b, 0, 0);
      w.qt = w.c - 1 - s.nctx;
      w.pair = s.run && w.qt >= 0 && w.qt * kTile < s.n;
      if (w.pair) {
        const int64_t g = gridDim.x;
        w.h = static_cast<int>(((static_cast<int64_t>(blockIdx.x) - w.n0) % g + g) % g);
      }
    }
  }
}

// Keys of key tile j of unit u (context tile or chunk tile).
__device__ __forceinline__ int tile_keys(const Unit& u, int j) {
  return j < u.nctx ? min(kTile, u.C - j * kTile) : min(kTile, u.n - (j - u.nctx) * kTile);
}

// 2^x by the hardware's approximate exponential (ex2.approx, relative error
// well below the 16-bit rounding p goes through next; inputs here are <= 8)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Round two p values to the 16-bit element type, packed low / high for P,
// and add the rounded values to the running sum.
__device__ __forceinline__ uint32_t pack2_16(float p0, float p1, float& sum, __nv_bfloat16*) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
  sum += __low2float(h) + __high2float(h);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack2_16(float p0, float p1, float& sum, __half*) {
  const __half2 h = __floats2half2_rn(p0, p1);
  sum += __low2float(h) + __high2float(h);
  return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace pf

// kcmap / vcmap: the caches as rows of head_dim (box 64 x BS, and a whole
// block slice-major); qmap / knmap / vnmap: q, k, v as (64, heads, T,
// head_dim / 64) with boxes (64, 1, 128, 1) for a q or key slice of 128
// rows and (64, 1, 16, head_dim / 64) for 16 value rows slice-major.
template <typename T, int D, int BS, bool kCost>
__global__ void __launch_bounds__(pf::kThreads, 1)
    pa_prefill_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap knmap,
                      const __grid_constant__ CUtensorMap vnmap,
                      const __grid_constant__ CUtensorMap kcmap,
                      const __grid_constant__ CUtensorMap vcmap, long long budget) {
  using namespace pf;
  using Lay = Layout<D>;
  constexpr int NST = Lay::kStages;
  constexpr int kSl = Lay::kSlices;
  constexpr int kVT = Lay::kVTokens;
  static_assert(D == 128 || D == 256, "head_dim");
  static_assert(BS % 16 == 0 && kTile % BS == 0 && kVT % BS == 0, "block size");
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;

  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (sm100::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* qs = smem;
  uint8_t* ring = smem + Lay::kRingOff;
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + Lay::kCtrlOff);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      sm100::mbar_init(&c.full[s], 1);
      sm100::mbar_init(&c.empty[s], 1);
    }
    sm100::mbar_init(&c.qfull, 1);
    sm100::mbar_init(&c.qempty, 1);
    sm100::mbar_init(&c.s_full[0], 1);
    sm100::mbar_init(&c.s_full[1], 1);
    sm100::mbar_init(&c.p_ready, kSoftmaxThreads);
    sm100::mbar_init(&c.o_done[0], 1);
    sm100::mbar_init(&c.o_done[1], 1);
    for (int p = 0; p < kProducers; ++p) sm100::mbar_init(&c.tail[p], 1);
    sm100::mbar_init(&c.drain, 1);
    sm100::mbar_init(&c.never, 1);
    c.abort = 0;
  }
  if (warp == kMmaWarp) {
    sm100::tmem_alloc(&c.tmem, kTmemCols);
    sm100::tmem_relinquish();
  }
  if (warp == kMmaWarp + 1 && lane == 0) {
    sm100::tma_prefetch_desc(&qmap);
    sm100::tma_prefetch_desc(&knmap);
    sm100::tma_prefetch_desc(&vnmap);
    sm100::tma_prefetch_desc(&kcmap);
    sm100::tma_prefetch_desc(&vcmap);
  }
  sm100::fence_proxy_async_smem();
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = c.tmem;
  volatile int* abort_flag = &c.abort;

  if (warp > kMmaWarp) {
    // ========================= producers ==========================================
    // Per unit: q, then keys of tile 0, then (keys of tile j, values of tile
    // j - 1) for j >= 1, then the last tile's values -- the order the MMA
    // warp consumes the ring in.  Every producer warp walks this sequence;
    // producer `pid` fills the stages g with g % kProducers == pid (and loads
    // q if pid == 0).
    const uint32_t pid = static_cast<uint32_t>(warp - kMmaWarp - 1);
    uint64_t* my_tail = &c.tail[pid];
    uint64_t keep;  // q, the chunk's keys / values and the context: read by several units
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(keep));
    uint32_t g = 0, un = 0, tn = 0;
    int tail_pending = -1;
    bool ok = true;

    // Block id of each lane's block in context tile j (lanes past the tile
    // or tiles past the context: -1, unused).  Loaded a tile ahead of its
    // use, so the table read's latency is hidden behind the current tile's
    // copies; ctx_row turns it into a TMA row only where it is used.
    auto ctx_id = [&](const Unit& u, int j) -> int32_t {
      if (j >= u.nctx || lane >= (tile_keys(u, j) + BS - 1) / BS) return -1;
      return __ldg(a.block_tables + static_cast<int64_t>(u.b) * a.max_blocks_per_seq +
                   j * (kTile / BS) + lane);
    };
    // TMA row of a block id; an id outside the pool becomes a negative row,
    // which TMA fills with zeros instead of reading memory.
    auto ctx_row = [&](const Unit& u, int32_t id) -> int32_t {
      const int kvh = u.h / a.group;
      return (id < 0 || id >= a.num_blocks) ? -BS : (id * a.num_kv_heads + kvh) * BS;
    };

    auto issue_k = [&](const Unit& u, int j, int32_t y) -> bool {
      const int kvh = u.h / a.group;
      const int nk = tile_keys(u, j);
      const bool ctx = j < u.nctx;
      const int nblk = (nk + BS - 1) / BS;
      for (int sl = 0; sl < kSl; ++sl, ++g) {
        if (g % kProducers != pid) continue;
        const int slot = g % NST;
        if (!__all_sync(0xffffffffu, sm100::mbar_wait(&c.empty[slot], ((g / NST) & 1) ^ 1, budget,
                                                        abort_flag)))
          return false;
        uint8_t* st = ring + slot * kStage;
        if (ctx) {
          if (lane == 0) sm100::mbar_arrive_expect_tx(&c.full[slot], nblk * BS * 128);
          __syncwarp();
          if (lane < nblk)
            sm100::tma_load_2d(st + lane * BS * 128, &kcmap, &c.full[slot], sl * 64, y, keep);
        } else {
          if (lane == 0) {
            sm100::mbar_arrive_expect_tx(&c.full[slot], kStage);
            sm100::tma_load_4d(st, &knmap, &c.full[slot], 0, kvh,
                               u.s0 + (j - u.nctx) * kTile, sl, keep);
          }
        }
        __syncwarp();
      }
      return true;
    };

    // Values of tile j.  The stage that holds the tile's last key, when that
    // key ends inside a 16-key MMA step, lands on the producer's own barrier
    // first and the rows past it are cleared (P is zero there, but 0 * NaN
    // would be NaN) before the stage is handed to the MMA warp.
    auto issue_v = [&](const Unit& u, int j, int32_t y) -> bool {
      const int kvh = u.h / a.group;
      const int nk = tile_keys(u, j);
      const bool ctx = j < u.nctx;
      const int vbs = ctx ? BS : 16;  // rows per copy (cache block / 16 chunk rows)
      const int nv = (nk + kVT - 1) / kVT;
      for (int v = 0; v < nv; ++v, ++g) {
        if (g % kProducers != pid) continue;
        const int slot = g % NST;
        if (!__all_sync(0xffffffffu, sm100::mbar_wait(&c.empty[slot], ((g / NST) & 1) ^ 1, budget,
                                                        abort_flag)))
          return false;
        const int toks = min(kVT, nk - v * kVT);
        const int ncp = (toks + vbs - 1) / vbs;  // copies in this stage
        const bool tail = v == nv - 1 && (nk % 16) != 0;
        uint64_t* land = tail ? my_tail : &c.full[slot];
        uint8_t* st = ring + slot * kStage;
        if (lane == 0) sm100::mbar_arrive_expect_tx(land, ncp * vbs * D * 2);
        __syncwarp();
        if (ctx) {
          const int jb0 = v * kVT / BS;
          const int32_t yj = __shfl_sync(0xffffffffu, y, (jb0 + lane) & 31);
          if (lane < ncp)
            sm100::tma_load_3d(st + lane * BS * D * 2, &vcmap, land, 0, yj, 0, keep);
        } else if (lane < ncp) {
          sm100::tma_load_4d(st + lane * 16 * D * 2, &vnmap, land, 0, kvh,
                             u.s0 + (j - u.nctx) * kTile + v * kVT + lane * 16, 0, keep);
        }
        __syncwarp();
        if (tail) {
          tail_pending = slot;
          if (!__all_sync(0xffffffffu, sm100::mbar_wait(my_tail, tn & 1, budget, abort_flag)))
            return false;
          ++tn;
          tail_pending = -1;
          const int r0 = toks;                  // first row past the tile's last key
          const int r1 = (r0 + 15) / 16 * 16;   // end of its 16-key step
          const int pieces = (r1 - r0) * kSl * 8;
          for (int i = lane; i < pieces; i += 32) {
            const int line = i / 8, piece = i % 8;
            const int r = r0 + line / kSl, sl = line % kSl;
            *reinterpret_cast<uint4*>(st + (r / vbs) * vbs * D * 2 + sl * vbs * 128 +
                                      (r % vbs) * 128 + piece * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          sm100::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) sm100::mbar_arrive(&c.full[slot]);
        }
      }
      return true;
    };

    Walk wk = walk_begin(a);
    Unit u;
    while (ok && walk_next<kCost>(a, wk, u)) {
      // q tile (rows past the chunk belong to other sequences or lie past T,
      // where TMA fills zeros; their rows are never stored)
      if (pid == 0) {
        ok = __all_sync(0xffffffffu, sm100::mbar_wait(&c.qempty, (un & 1) ^ 1, budget, abort_flag));
        if (!ok) break;
        if (lane == 0) sm100::mbar_arrive_expect_tx(&c.qfull, kSl * kStage);
        __syncwarp();
        if (lane < kSl)
          sm100::tma_load_4d(qs + lane * kStage, &qmap, &c.qfull, 0, u.h, u.s0 + u.qt * kTile, lane,
                             keep);
        ++un;
      }
      int32_t yprev = 0;
      int32_t id = ctx_id(u, 0);
      for (int j = 0; j < u.ntiles && ok; ++j) {
        const int32_t y = j < u.nctx ? ctx_row(u, id) : 0;
        id = ctx_id(u, j + 1);  // next tile's ids, first used in the next iteration
        ok = issue_k(u, j, y);
        if (ok && j > 0) ok = issue_v(u, j - 1, yprev);
        yprev = y;
      }
      if (ok) ok = issue_v(u, u.ntiles - 1, yprev);
    }
    if (!ok) {
      if (lane == 0) c.abort = 1;
      // copies already issued must land before the CTA may exit
      for (uint32_t gg = g > NST ? g - NST : 0; gg < g; ++gg)
        if (gg % kProducers == pid && static_cast<int>(gg % NST) != tail_pending)
          sm100::mbar_wait(&c.full[gg % NST], (gg / NST) & 1, budget, nullptr);
      if (tail_pending >= 0) sm100::mbar_wait(my_tail, tn & 1, budget, nullptr);
      if (un > 0) sm100::mbar_wait(&c.qfull, (un - 1) & 1, budget, nullptr);
    }
  } else if (warp == kMmaWarp) {
    // ========================= MMA issuer =========================================
    // The whole warp runs the loop in convergent code; one elected lane
    // issues each MMA and commit.  Per unit: QK^T(0), then (QK^T(j),
    // P.V(j - 1)) for j >= 1, then P.V(last), so the next tile's logits are
    // computed while the softmax warps work on this tile's.
    constexpr unsigned kAll = 0xffffffffu;
    constexpr uint32_t id_qk = sm100::idesc_f16(kBf16, false, false, 128, kTile);
    constexpr uint32_t id_pv = sm100::idesc_f16(kBf16, false, true, 128, D);
    const uint32_t q_base = sm100::smem_u32(qs);
    const uint32_t ring_base = sm100::smem_u32(ring);
    uint32_t g = 0, un = 0, gt = 0, pn = 0;
    bool ok = true;
    if (a.selftest_stall) ok = __all_sync(kAll, sm100::mbar_wait(&c.never, 0, budget, abort_flag));

    auto qk = [&]() -> bool {
      const uint32_t sbuf = tmem + ((gt & 1) ? kS1Col : 0);
      for (int sl = 0; sl < kSl; ++sl) {
        const int slot = g % NST;
        if (!__all_sync(kAll, sm100::mbar_wait(&c.full[slot], (g / NST) & 1, budget, abort_flag)))
          return false;
        sm100::tc_fence_after();
        const uint32_t st = ring_base + slot * kStage;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = sm100::smem_desc(q_base + sl * kStage + kk * 32, 16, 1024, sm100::kSw128);
          const uint64_t bd = sm100::smem_desc(st + kk * 32, 16, 1024, sm100::kSw128);
          sm100::mma_f16_elect(sbuf, ad, bd, id_qk, (sl | kk) != 0);
        }
        sm100::mma_commit_elect(&c.empty[slot]);
        ++g;
      }
      return true;
    };
    auto pv = [&](const Unit& u, int j) -> bool {
      if (!__all_sync(kAll, sm100::mbar_wait(&c.p_ready, pn & 1, budget, abort_flag))) return false;
      const uint32_t pb = pn & 1;  // logits buffer of this tile, which now holds its P
      ++pn;
      sm100::tc_fence_after();
      const int nk = tile_keys(u, j);
      const int vbs = j < u.nctx ? BS : 16;
      const int nv = (nk + kVT - 1) / kVT;
      for (int v = 0; v < nv; ++v) {
        const int slot = g % NST;
        if (!__all_sync(kAll, sm100::mbar_wait(&c.full[slot], (g / NST) & 1, budget, abort_flag)))
          return false;
        sm100::tc_fence_after();
        const uint32_t st = ring_base + slot * kStage;
        const int toks = min(kVT, nk - v * kVT);
        for (int r = 0; r < toks; r += 16) {
          const int key = v * kVT + r;
          // P of keys 64 * h .. 64 * h + 63 is in columns 64 * h .. 64 * h + 31
          // of the tile's logits buffer, two keys per 32-bit column
          const uint32_t at = tmem + (pb ? kS1Col : 0) + (key / 64) * 64 + (key % 64) / 2;
          const uint64_t bd = sm100::smem_desc(st + (r / vbs) * vbs * D * 2 + (r % vbs) * 128,
                                               vbs * 128, 1024, sm100::kSw128);
          sm100::mma_f16_ts_elect(tmem + kOCol, at, bd, id_pv, (j | v | r) != 0);
        }
        sm100::mma_commit_elect(&c.empty[slot]);
        ++g;
      }
      sm100::mma_commit_elect(&c.o_done[pb]);
      return true;
    };

    Walk wk = walk_begin(a);
    Unit u;
    while (ok && walk_next<kCost>(a, wk, u)) {
      ok = __all_sync(kAll, sm100::mbar_wait(&c.qfull, un & 1, budget, abort_flag));
      if (!ok) break;
      ++un;
      sm100::tc_fence_after();
      for (int j = 0; j < u.ntiles && ok; ++j) {
        ok = qk();
        if (!ok) break;
        if (j == u.ntiles - 1) sm100::mma_commit_elect(&c.qempty);
        sm100::mma_commit_elect(&c.s_full[gt & 1]);
        ++gt;
        if (j > 0) ok = pv(u, j - 1);
      }
      if (ok) ok = pv(u, u.ntiles - 1);
    }
    if (!ok) {
      if (lane == 0) c.abort = 1;
      // no MMA may still be running when tensor memory is released
      sm100::mma_commit_elect(&c.drain);
      sm100::mbar_wait(&c.drain, 0, budget, nullptr);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ========================= softmax + epilogue (warps 0-7) =====================
    // Thread (half, r) owns query row r of the unit (tensor-memory lane r) and
    // keys 64 * half .. 64 * half + 63 of every tile, head_dim columns
    // half * D / 2 .. of the output.  Per tile, half 1 publishes its partial
    // max, half 0 forms the row's reference max (moving it lazily) and
    // publishes it, and half 1 adopts it, so both halves scale their
    // probabilities by the same reference.  Every softmax thread runs the same
    // iterations and barriers whatever happens; a failed wait only marks the
    // abort, which ends later waits.
    const int half = tid >> 7;
    const int r = tid & 127;
    const int k0 = half * (kTile / 2);  // first key column of this half
    const int d0 = half * (D / 2);      // first output column of this half
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = a.scale_log2;
    auto pair_sync = [] { asm volatile("bar.sync 1, 256;" ::: "memory"); };
    uint32_t gt = 0;  // key tiles so far (logits buffer, s_full / o_done phases)
    Walk wk = walk_begin(a);
    Unit u;
    while (walk_next<kCost>(a, wk, u)) {
      const int i = u.qt * kTile + r;  // this row's place in the chunk
      const bool row_ok = i < u.n;
      float m_ref = -INFINITY, lsum = 0.f;
      bool bad = u.poison;
      for (int j = 0; j < u.ntiles; ++j, ++gt) {
        const int nk = tile_keys(u, j);
        const bool ctx = j < u.nctx;
        // visible keys of the tile form a prefix: all context keys, chunk keys
        // up to the row's own
        const int vis = ctx ? nk : max(0, min(nk, i - (j - u.nctx) * kTile + 1));
        // context block ids: one outside the pool poisons the unit.  The id is
        // loaded here and tested after this tile's P is written, so the load's
        // latency is not on the softmax's path.
        int32_t blk_id = 0;
        if (ctx && lane < (nk + BS - 1) / BS)
          blk_id = __ldg(a.block_tables + static_cast<int64_t>(u.b) * a.max_blocks_per_seq +
                         j * (kTile / BS) + lane);
        if (!sm100::mbar_wait(&c.s_full[gt & 1], (gt >> 1) & 1, budget, abort_flag)) c.abort = 1;
        sm100::tc_fence_after();
        __syncwarp();
        const uint32_t sbuf = tmem + lane_base + ((gt & 1) ? kS1Col : 0);
        float mx = -INFINITY;
#pragma unroll 1
        for (int c0 = k0; c0 < k0 + kTile / 2; c0 += 32) {
          float sv[32];
          sm100::tmem_ld16(sbuf + c0, *reinterpret_cast<float(*)[16]>(&sv[0]));
          sm100::tmem_ld16(sbuf + c0 + 16, *reinterpret_cast<float(*)[16]>(&sv[16]));
          sm100::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c0 + e < vis) mx = fmaxf(mx, sv[e]);
        }
        // the row's reference max, agreed by both halves
        if (half == 1) c.xrow[r] = mx;
        pair_sync();
        float corr = 1.f;
        bool move = false;
        if (half == 0) {
          const float mt = fmaxf(mx, c.xrow[r]) * sl2;
          const float m_new = fmaxf(m_ref, mt);
          move = m_new > m_ref + kRescaleLog2;
          if (move) {
            corr = m_ref == -INFINITY ? 0.f : exp2f(m_ref - m_new);
            m_ref = m_new;
          }
          c.xrow[r] = m_ref;
        }
        pair_sync();
        if (half == 1) {
          const float m_new = c.xrow[r];
          move = m_new != m_ref;
          if (move) {
            corr = m_ref == -INFINITY ? 0.f : exp2f(m_ref - m_new);
            m_ref = m_new;
          }
        }
        if (move) lsum *= corr;
        const bool rescale = j > 0 && __any_sync(0xffffffffu, move);
        if (rescale) {
          // O must be complete up to the previous tile before it is rescaled
          if (!sm100::mbar_wait(&c.o_done[(gt - 1) & 1], ((gt - 1) >> 1) & 1, budget, abort_flag))
            c.abort = 1;
          sm100::tc_fence_after();
          __syncwarp();
          // the warp's rows that moved their reference max rescale their half of the O row
#pragma unroll 1
          for (int c0 = d0; c0 < d0 + D / 2; c0 += 16) {
            float ov[16];
            sm100::tmem_ld16(tmem + lane_base + kOCol + c0, ov);
            sm100::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] *= corr;
            sm100::tmem_st16(tmem + lane_base + kOCol + c0, ov);
          }
          sm100::tmem_wait_st();
        }
        // p = 2^(s * scale * log2(e) - m_ref) for the visible keys, rounded to
        // 16 bits and packed two keys per 32-bit column into this half's first
        // 32 logit columns (keys k0 + 2c, k0 + 2c + 1 -> column k0 + c), over
        // logits this thread has already read.  The P.V that reads P is issued
        // before the MMA that next writes this buffer (the QK^T two tiles on),
        // and the tensor core runs them in order.
        const float neg_m = -m_ref;
#pragma unroll 1
        for (int c0 = k0; c0 < k0 + kTile / 2; c0 += 32) {
          float sv[32];
          sm100::tmem_ld16(sbuf + c0, *reinterpret_cast<float(*)[16]>(&sv[0]));
          sm100::tmem_ld16(sbuf + c0 + 16, *reinterpret_cast<float(*)[16]>(&sv[16]));
          sm100::tmem_wait_ld();
          float w[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = c0 + e < vis ? ex2_approx(fmaf(sv[e], sl2, neg_m)) : 0.f;
            const float p1 = c0 + e + 1 < vis ? ex2_approx(fmaf(sv[e + 1], sl2, neg_m)) : 0.f;
            w[e / 2] = __uint_as_float(pack2_16(p0, p1, lsum, static_cast<T*>(nullptr)));
          }
          sm100::tmem_st16(sbuf + k0 + (c0 - k0) / 2, w);
        }
        sm100::tmem_wait_st();
        sm100::tc_fence_before();
        sm100::mbar_arrive(&c.p_ready);
        if (ctx) bad |= __any_sync(0xffffffffu, blk_id < 0 || blk_id >= a.num_blocks);
      }
      // ---- epilogue of the unit: O / (both halves' sums) into out ------------------
      if (half == 1) c.xrow[r] = lsum;
      pair_sync();
      float total = lsum;
      if (half == 0) {
        total = lsum + c.xrow[r];
        c.xrow[r] = total;
      }
      pair_sync();
      if (half == 1) total = c.xrow[r];
      pair_sync();  // xrow is free for the next unit's first tile
      if (!sm100::mbar_wait(&c.o_done[(gt - 1) & 1], ((gt - 1) >> 1) & 1, budget, abort_flag))
        c.abort = 1;
      sm100::tc_fence_after();
      __syncwarp();
      const bool poison = bad || *abort_flag != 0;
      const float inv = 1.f / total;
      const int64_t orow = (static_cast<int64_t>(u.s0) + i) * a.num_heads + u.h;
#pragma unroll 1
      for (int c0 = d0; c0 < d0 + D / 2; c0 += 16) {
        float ov[16];
        sm100::tmem_ld16(tmem + lane_base + kOCol + c0, ov);
        sm100::tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 16; ++e) ov[e] = poison ? qnan() : ov[e] * inv;
          store_row16(a.out, orow * D + c0, a.out_dtype, ov);
        }
      }
      sm100::tc_fence_before();
    }
  }

  // ---- teardown -------------------------------------------------------------------
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  if (warp == kMmaWarp) sm100::tmem_dealloc(tmem, kTmemCols);
}

// Persistent launch: one CTA per SM (the kernel takes ~226 KB of shared
// memory and all 512 tensor-memory columns), at most one per unit.
template <typename T, int D, int BS>
cudaError_t launch_prefill_t(const PrefillArgs& a, const CUtensorMap (&m)[5], int num_sms,
                             cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  auto kern = a.cost_levels > 0 ? pa_prefill_kernel<T, D, BS, true>
                                 : pa_prefill_kernel<T, D, BS, false>;
  // set once per device; concurrent first calls set the same attributes
  static std::atomic<bool> configured[128];
  if (!configured[dev].load(std::memory_order_acquire)) {
    for (auto k : {pa_prefill_kernel<T, D, BS, true>, pa_prefill_kernel<T, D, BS, false>}) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           pf::Layout<D>::kSmem);
      if (e != cudaSuccess) return e;
    }
    configured[dev].store(true, std::memory_order_release);
  }
  const int64_t units = static_cast<int64_t>(a.qtiles) * a.num_seqs * a.num_heads;
  if (units == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(units, num_sms));
  const long long budget = a.selftest_stall ? pf::kSelftestBudget : pf::kWaitBudget;
  kern<<<grid, pf::kThreads, pf::Layout<D>::kSmem, s>>>(a, m[0], m[1], m[2], m[3], m[4], budget);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefill_dtype(const PrefillArgs& a, const CUtensorMap (&m)[5], int num_sms,
                                 cudaStream_t s) {
  if (a.head_dim == 256 && a.block_size == 16) return launch_prefill_t<T, 256, 16>(a, m, num_sms, s);
  if (a.head_dim == 256 && a.block_size == 32) return launch_prefill_t<T, 256, 32>(a, m, num_sms, s);
  if (a.head_dim == 128 && a.block_size == 16) return launch_prefill_t<T, 128, 16>(a, m, num_sms, s);
  if (a.head_dim == 128 && a.block_size == 32) return launch_prefill_t<T, 128, 32>(a, m, num_sms, s);
  if (a.head_dim == 128 && a.block_size == 64) return launch_prefill_t<T, 128, 64>(a, m, num_sms, s);
  return cudaErrorInvalidValue;
}

}  // namespace pa
