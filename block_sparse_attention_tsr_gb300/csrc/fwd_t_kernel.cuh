// fwd_t_kernel.cuh -- the block-sparse attention forward kernel in the key-major
// (transposed) tile orientation, d = 128; host side in fwd.cu, instantiations
// in fwd_t.cu.
//
// The plan gives one work item per 64-row query block and, for it, a list of
// 64 x 64 tiles (64 queries x 64 keys: contiguous key blocks, or 64 gathered
// keys of the block's key list).  The kernel takes the list two tiles at a time:
// one step computes, for 128 keys (two arbitrary 64-key tiles of the list) and
// the block's 64 queries,
//
//     S^T = K Q^T           tcgen05, M = 128 keys, N = 64 queries, K = d
//     P^T = exp(S^T - m)    per key lane in TMEM, P^T to shared memory (bf16)
//     O^T += V^T P^T        tcgen05, M = d = 128, N = 64 queries, K = 128 keys
//
// so a query block's work is exactly its own key blocks: a 64-row block is
// never widened to 128 rows to fit the tensor core's M = 128 side (Tessera
// abstract: physical tiles chosen by mask shape, here subdividing the 128-row
// tile; FG-Attn abstract: skipping at 64-query x 1-key slice granularity).
//
// One CTA per SM works on one item at a time, 384 threads:
//   warp 0      K producer: the item's 64-row query tile, then per step its two
//               64-key tiles of K, by TMA, or by row gathers for key lists and
//               temporal-major items; step j goes to slot j & 1
//   warp 2      V producer: the same for V; V loads wait for PVs, so they run
//               in a warp of their own and never hold up K
//   warps 1, 11 MMA issuers (one thread each), one per softmax group: QK of the
//               group's step t, then PV of its step t - 1.  One issuing thread
//               leaves the tensor pipe idle whenever it waits on a barrier (its
//               queue holds only a few MMAs); two keep it fed
//   warps 3..6  softmax group 0: the item's even steps
//   warps 7..10 softmax group 1: the item's odd steps
// Each group keeps its own running maximum, row sums, two P^T buffers and O^T
// accumulator (split of the item's key list in two, so the two groups'
// softmax work overlaps); the epilogue merges the two halves of the item
// (the split-KV combine: O = (a0 O0 + a1 O1) / (a0 l0 + a1 l1) with
// a_g = 2^(m_g - max(m0, m1))) and stores O and lse.
//
// Softmax in the transposed layout.  A thread holds one key's logits for the
// 64 queries, so reductions over keys run across the 128 threads of a group.
// The running maximum per query is therefore not taken every step: P^T is
// computed against a per-query reference m (shared memory), and only when an
// exponent y - m (base 2) exceeds 16 -- a logit 2^16 times its reference --
// does the group take the exact column maximum of the step (warp shuffles +
// shared memory), raise m, rewrite the step's P^T and rescale its row sums and
// O^T by 2^(m_old - m_new).  A warp adds a half-step's P to its row-sum shares
// only when none of its exponents is above 16, so the correction knows which
// optimistic values it has to take back.  The first step of every item starts
// from m = -1e30, so it always takes the exact path.  Every thread keeps its
// key's share of the 64 row sums in TMEM; the shares are summed over the 128
// threads once per item, in the epilogue.  The result is the same masked
// softmax; only the reference point of the exponentials differs, which cancels
// in O = (sum_k P V) / (sum_k P).
#pragma once
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstddef>
#include <cmath>
#include <cstring>

#include "fwd_kernel.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tsr {
namespace fwd_t {

using fwd::FwdParamsT;
using fwd::kModeList;
using fwd::kModePerm;
using fwd::kModeTma;
using fwd::ReqParams;

constexpr int D = 128;                 // head dimension of this kernel
constexpr int QB = 64;                 // query rows per item
constexpr int KT = 64;                 // keys per plan tile (two per step)
constexpr int KS = 2, VS = 2;          // K and V slots: slot g feeds group g's steps
constexpr int kThreads = 384;
constexpr float kFixThreshold = 16.0f; // base-2 units above the reference maximum
constexpr float kMrefInit = -1.0e30f;  // reference maximum of a query with no key yet
constexpr float kLn2 = 0.69314718055994530942f;

// Shared-memory layout (dynamic, 1024-byte aligned).  Q tile: [d chunk (2)]
// [64 rows][128 B]; K / V slots: [d chunk (2)][128 rows][128 B] (rows 0..63 the
// step's first tile, 64..127 its second); P^T, two per group (the group's
// consecutive steps alternate): [128 keys][128 B] (64 queries); all in the
// 128-byte swizzled layout (16-byte unit u of row r at u ^ (r & 7)).  The
// epilogue stages the item's O in group 0's first P^T buffer.
constexpr int Q_BYTES = QB * D * 2;                  // 16 KB
constexpr int KV_BYTES = 2 * KT * D * 2;             // 32 KB
constexpr int P_BYTES = 2 * KT * QB * 2;             // 16 KB
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + Q_BYTES;
constexpr int OFF_V = OFF_K + KS * KV_BYTES;
constexpr int OFF_P = OFF_V + VS * KV_BYTES;
constexpr int SMEM_BYTES = OFF_P + 4 * P_BYTES + 1024;   // + alignment slack
static_assert(SMEM_BYTES <= 220 * 1024, "shared memory");

// TMEM columns: per group S^T double buffer (2 x 64) and O^T (64), then each
// group's row-sum shares (64).
constexpr int TM_GROUP = 192;
constexpr int TM_O = 128;
constexpr int TM_L = 384;
constexpr uint32_t IDESC_QK = idesc_bf16(128, QB, false, false);   // A = K (K-major), B = Q (K-major)
constexpr uint32_t IDESC_PV = idesc_bf16(128, QB, true, true);     // A = V^T (MN-major), B = P^T (MN-major)

struct alignas(16) CtrlT {
  uint64_t q_full, q_empty;
  uint64_t k_full[KS], k_empty[KS], v_full[VS], v_empty[VS];
  // per group and P^T buffer: a group's next arrival on the same buffer waits
  // for the PV of that buffer's previous step, so no barrier runs two phases
  // ahead of its waiter
  uint64_t s_full[2][2], p_full[2][2], pv_done[2][2], o_full, o_empty;
  uint64_t item_full[2], item_empty[2];
  uint64_t grp[2], pair;
  uint64_t final_bar[2], never;
  int32_t item_slot[2];
  int32_t fixflag[2][2];
  alignas(16) float mref[2][QB];   // read as float4 by the softmax
  alignas(16) float mold[2][QB];   // the reference before the last raise (correction path)
  float alpha[2][QB];
  float red[2][4][QB];
  float lsum[2][QB];
  float fac[2][QB];           // epilogue: each group's factor a_g / l per query
  float lse2[QB];             // epilogue: lse in base-2 units, or -inf
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t split_last;         // split-KV: this CTA's unit was the last part of its item
};

// The softmax reads 4 reference maxima at a time (16-byte loads).
static_assert(offsetof(CtrlT, mref) % 16 == 0 && offsetof(CtrlT, mold) % 16 == 0,
              "reference maxima must be 16-byte aligned");

__device__ __forceinline__ int32_t unpermute(int32_t tp, int32_t F, int32_t S) {
  return (tp % F) * S + tp / F;
}

// Bits [lo, hi) of a 64-bit mask as two words (0 <= lo <= hi <= 64).
__device__ __forceinline__ void range64(uint32_t& w0, uint32_t& w1, int lo, int hi) {
  auto word = [](int a, int b) -> uint32_t {   // bits [a, b) of one word, 0 <= a <= b <= 32
    const uint32_t hi_m = (b >= 32) ? 0xFFFFFFFFu : ((1u << b) - 1u);
    const uint32_t lo_m = (a >= 32) ? 0xFFFFFFFFu : ((1u << a) - 1u);
    return a < b ? (hi_m & ~lo_m) : 0u;
  };
  w0 |= word(min(lo, 32), min(hi, 32));
  w1 |= word(max(lo - 32, 0), max(hi - 32, 0));
}

__device__ __forceinline__ uint32_t dbyte(const uint4& a, const uint4& b, int i) {
  return fwd::desc_byte(a, b, i);
}

// y = x * s + c for two lanes at once (fma.rn.f32x2), c per lane.
__device__ __forceinline__ void fma2c(float& y0, float& y1, float x0, float x1, float s, float c0,
                                      float c1) {
  asm("{\n\t.reg .b64 xa, sa, ca;\n\tmov.b64 xa, {%2, %3};\n\tmov.b64 sa, {%4, %4};\n\t"
      "mov.b64 ca, {%5, %6};\n\tfma.rn.f32x2 xa, xa, sa, ca;\n\tmov.b64 {%0, %1}, xa;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(s), "f"(c0), "f"(c1));
}

// Copy 64 rows of d = 128 bf16 values (row r from source row src(r) of a head)
// into a tile region in the 128-byte swizzled K-major layout: row r of d chunk
// c at dst + c * chunk_stride + r * 128 (the region's rows start at an 8-row
// boundary, so r & 7 is the row's position in its swizzle atom).  Each lane
// copies 32 16-byte units; `rows` holds the source rows of tile rows lane and
// lane + 32.  Completion is tied to the phase by the caller (cp.async arrive).
__device__ __forceinline__ void gather64(const __nv_bfloat16* head_base, const int32_t (&rows)[2],
                                         uint32_t dst, uint32_t chunk_stride, int lane) {
#pragma unroll
  for (int m = 0; m < 32; ++m) {
    const int row = 2 * m + (lane >> 4);                  // 16 units per row
    const int src = __shfl_sync(0xFFFFFFFFu, rows[m >> 4], row & 31);   // row >> 5 == m >> 4
    const int j = lane & 15, c = j >> 3, u = j & 7;
    const void* g = reinterpret_cast<const uint8_t*>(head_base + static_cast<size_t>(src) * D) + j * 16;
    cp_async_16(dst + c * chunk_stride + row * 128 + ((u ^ (row & 7)) << 4), g);
  }
}

// In-warp transposed reduction of NV (32 or 64) values per lane: after it,
// lane l holds the reduction over the warp's 32 lanes of entry l (NV = 32) in
// v[0], or of entries 2l and 2l + 1 (NV = 64) in v[0], v[1].
template <bool MAX, int NV>
__device__ __forceinline__ void warp_reduce(float (&v)[NV], int lane) {
#pragma unroll
  for (int s = 0; s < 5; ++s) {
    const int o = 16 >> s, H2 = (NV >> s) / 2;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < NV / 2; ++i) {
      if (i < H2) {
        const float send = up ? v[i] : v[i + H2];
        const float keep = up ? v[i + H2] : v[i];
        const float got = __shfl_xor_sync(0xFFFFFFFFu, send, o);
        v[i] = MAX ? fmaxf(keep, got) : keep + got;
      }
    }
  }
}

// K or V of one step of an item: its two 64-key tiles into a ring slot
// ([d chunk][128 rows][128 B], the first tile in rows 0..63).  TMA for
// contiguous tiles (a missing second tile reads rows past N, which TMA fills
// with zeros); row gathers for key lists (rows named by gidx; a missing
// second tile repeats the first tile's rows) and temporal-major items (rows
// through the inverse permutation; rows past N read row 0).  Gathered rows
// complete on the barrier through cp.async arrive plus lane 0's arrival.
// The item's plan entries held in a producer warp's lanes, one 32-entry chunk
// ahead of use: lane l holds entry begin + 32 c + l of the current chunk c and
// of chunk c + 1.  A step's two key tiles are then read with shuffles, and the
// load of the next chunk is issued 16 steps before it is needed, so no copy
// waits behind a dependent global load.  All 32 lanes call every member.
struct EntryWindow {
  int32_t cur, nxt, chunk;
  __device__ __forceinline__ void start(const ReqParams& rq, int32_t begin, int32_t n, int lane) {
    chunk = 0;
    cur = lane < n ? __ldg(&rq.entries[begin + lane]).x : 0;
    nxt = 32 + lane < n ? __ldg(&rq.entries[begin + 32 + lane]).x : 0;
  }
  // Key block of tile t (t = 2 * step + h); steps advance one at a time.
  __device__ __forceinline__ int32_t tile(const ReqParams& rq, int32_t begin, int32_t n, int32_t t,
                                          int lane) {
    const int32_t c = t >> 5;
    if (c != chunk) {
      chunk = c;
      cur = nxt;
      const int32_t e = 32 * (c + 1) + lane;
      nxt = e < n ? __ldg(&rq.entries[begin + e]).x : 0;
    }
    return __shfl_sync(0xFFFFFFFFu, cur, t & 31);
  }
};

// The two key tiles of step `step`: kv0, and kv1 for the second (a missing
// second tile: rq.N for TMA, which then reads rows past N as zeros; the first
// tile again for gathers).
__device__ __forceinline__ void step_tiles(EntryWindow& win, const ReqParams& rq, int32_t begin,
                                           int32_t n, int32_t step, bool gath, int lane,
                                           int32_t& kv0, int32_t& kv1) {
  kv0 = win.tile(rq, begin, n, 2 * step, lane);
  const int32_t t1 = win.tile(rq, begin, n, 2 * step + 1, lane);
  kv1 = (2 * step + 1 < n) ? t1 : (gath ? kv0 : rq.N);
}

// Source rows of a gathered step, tile h rows lane and lane + 32 in rows[h]:
// key-list rows named by gidx, or temporal-major rows through the inverse
// permutation (rows past N read row 0).
template <bool GATHER>
__device__ __forceinline__ void step_rows(const ReqParams& rq, int32_t kv0, int32_t kv1, int lane,
                                          int32_t (&rows)[2][2]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int32_t kv = h ? kv1 : kv0;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      if (GATHER) {
        rows[h][m] = __ldg(rq.gidx + kv + 32 * m + lane);
      } else {
        const int32_t tp = kv + 32 * m + lane;
        rows[h][m] = tp < rq.N ? unpermute(tp, rq.F, rq.S) : 0;
      }
    }
  }
}

// One step's K (or V) rows for the two key tiles into a ring slot
// ([d chunk][128 rows][128 B], the first tile in rows 0..63): TMA for
// contiguous tiles, row gathers (rows from step_rows) for key lists and
// temporal-major items.  Gathered rows complete on the barrier through
// cp.async arrive plus lane 0's arrival.
__device__ __forceinline__ void load_kv_step(bool gath, int32_t bh, int32_t N, int32_t kv0, int32_t kv1,
                                             const int32_t (&rows)[2][2], const CUtensorMap* map,
                                             const __nv_bfloat16* src, uint32_t dst, uint32_t bar,
                                             int lane) {
  if (gath) {
    const __nv_bfloat16* head = src + static_cast<size_t>(bh) * N * D;
    gather64(head, rows[0], dst, 2 * KT * 128, lane);
    gather64(head, rows[1], dst + KT * 128, 2 * KT * 128, lane);
    cp_async_arrive(bar);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  } else if (lane == 0) {
    mbar_arrive_expect_tx(bar, KV_BYTES);
    for (int h = 0; h < 2; ++h)
      for (int c = 0; c < 2; ++c)
        tma_load_3d(dst + c * (2 * KT * 128) + h * KT * 128, map, bar, c * 64, h ? kv1 : kv0, bh);
  }
}

// The K or V stream of one item, steps [0, ns): step j goes to slot j & 1, the
// slot of the group that consumes it (group j & 1), so each slot is a channel
// between the producer and one MMA issuer; cnt[s] counts the loads into slot s.
// The next step's tiles (and, for gathers, its source rows) are read while the
// current step's slot is awaited.  Returns false when a wait gave up.
template <bool GATHER, bool PERM, typename WaitFn>
__device__ __forceinline__ bool stream_item(const ReqParams& rq, int32_t bh, int32_t begin, int32_t n,
                                            int32_t layout, int32_t ns, const CUtensorMap* map,
                                            const __nv_bfloat16* src, uint32_t ring, uint64_t* full,
                                            uint64_t* empty, uint32_t (&cnt)[2], int site, int lane,
                                            WaitFn&& wait) {
  const bool gath = GATHER || (PERM && layout != 0);
  EntryWindow win;
  win.start(rq, begin, n, lane);
  int32_t kv0, kv1, rows[2][2] = {{0, 0}, {0, 0}};
  step_tiles(win, rq, begin, n, 0, gath, lane, kv0, kv1);
  if (gath) step_rows<GATHER>(rq, kv0, kv1, lane, rows);
  for (int32_t i = 0; i < ns; ++i) {
    const int s = i & 1;
    if (!wait(smem_u32(&empty[s]), (cnt[s] & 1) ^ 1, site)) return false;
    load_kv_step(gath, bh, rq.N, kv0, kv1, rows, map, src, ring + s * KV_BYTES, smem_u32(&full[s]), lane);
    ++cnt[s];
    if (i + 1 < ns) {
      step_tiles(win, rq, begin, n, i + 1, gath, lane, kv0, kv1);
      if (gath) step_rows<GATHER>(rq, kv0, kv1, lane, rows);
    }
  }
  return true;
}

template <int MODE, int MAXR>
__global__ void __launch_bounds__(kThreads, 1) bsa_fwd_t_kernel(const __grid_constant__ FwdParamsT<MAXR> p) {
  constexpr bool GATHER = MODE == kModeList;
  constexpr bool PERM = MODE == kModePerm;
  extern __shared__ uint8_t smem_raw[];
  __shared__ CtrlT ctrl;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* smem_gen = smem_raw + (base - smem_u32(smem_raw));   // generic pointer to `base`
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int32_t* abort_flag = &ctrl.abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctrl.q_full), 1);
    mbar_init(smem_u32(&ctrl.q_empty), 2);                // both MMA issuers
    for (int s = 0; s < KS; ++s) {
      mbar_init(smem_u32(&ctrl.k_full[s]), 1);
      mbar_init(smem_u32(&ctrl.k_empty[s]), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(smem_u32(&ctrl.v_full[s]), 1);
      mbar_init(smem_u32(&ctrl.v_empty[s]), 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(smem_u32(&ctrl.s_full[g][0]), 1);
      mbar_init(smem_u32(&ctrl.s_full[g][1]), 1);
      mbar_init(smem_u32(&ctrl.p_full[g][0]), 4);
      mbar_init(smem_u32(&ctrl.p_full[g][1]), 4);
      mbar_init(smem_u32(&ctrl.pv_done[g][0]), 1);
      mbar_init(smem_u32(&ctrl.pv_done[g][1]), 1);
      mbar_init(smem_u32(&ctrl.grp[g]), 4);
      ctrl.fixflag[g][0] = ctrl.fixflag[g][1] = -1;
      mbar_init(smem_u32(&ctrl.item_full[g]), 1);
      mbar_init(smem_u32(&ctrl.item_empty[g]), 11);  // 2 MMA issuers, V producer, 8 softmax warps
      mbar_init(smem_u32(&ctrl.final_bar[g]), 1);
    }
    mbar_init(smem_u32(&ctrl.o_full), 2);                 // both MMA issuers
    mbar_init(smem_u32(&ctrl.o_empty), 8);
    mbar_init(smem_u32(&ctrl.pair), 8);
    mbar_init(smem_u32(&ctrl.never), 1);
    ctrl.abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 2 * QB) ctrl.mref[threadIdx.x / QB][threadIdx.x % QB] = kMrefInit;
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctrl.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl.tmem_base;
  // Bounded wait on an mbarrier phase; the wait that times out first records
  // its site (bit 8 + site of the error word) next to DEV_ERR_TIMEOUT.
  auto wait = [&](uint32_t bar, uint32_t parity, int site) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (mbar_try_wait(bar, parity)) return true;
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        *abort_flag = 1;
        atomicOr(p.err, DEV_ERR_TIMEOUT | (1u << (8 + site)));
        return false;
      }
    }
  };

  if (warp == 0) {
    // ---------------------------------------------------------- K producer
    if (lane == 0) {
      tma_prefetch_desc(&p.req[0].tq);
      tma_prefetch_desc(&p.req[0].tk);
      tma_prefetch_desc(&p.req[0].tv);
    }
    uint32_t kc[2] = {0u, 0u}, qc = 0, seq = 0;
    bool ok = true;
    while (ok) {
      int32_t it = 0;
      if (lane == 0) it = atomicAdd(p.counter, 1);
      it = __shfl_sync(0xFFFFFFFFu, it, 0);
      const bool fin = it >= p.n_items;
      const int slot = seq & 1;
      if (!wait(smem_u32(&ctrl.item_empty[slot]), ((seq >> 1) & 1) ^ 1, 0)) break;
      if (lane == 0) {
        ctrl.item_slot[slot] = fin ? -1 : it;
        mbar_arrive(smem_u32(&ctrl.item_full[slot]));
      }
      ++seq;
      if (fin) break;
      const ReqParams& rq = p.req[fwd::req_of(p, it)];
      const int32_t li = it - rq.item_begin;
      const int4 i0 = __ldg(&rq.items[2 * li]);
      const int4 i1 = __ldg(&rq.items[2 * li + 1]);
      const int32_t bh = i0.x, qb = i0.y, begin = i0.z, n = i0.w - i0.z, layout = i1.x;
      const int32_t ns = (n + 1) >> 1;
      if (ns == 0) continue;
      // the query tile
      if (!wait(smem_u32(&ctrl.q_empty), (qc & 1) ^ 1, 1)) break;
      ++qc;
      {
        const uint32_t bar = smem_u32(&ctrl.q_full);
        if (PERM && layout != 0) {
          int32_t rows[2];
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int32_t tp = qb * QB + 32 * m + lane;
            rows[m] = tp < rq.N ? unpermute(tp, rq.F, rq.S) : 0;
          }
          gather64(rq.qg + static_cast<size_t>(bh) * rq.N * D, rows, base + OFF_Q, QB * 128, lane);
          cp_async_arrive(bar);
          __syncwarp();
          if (lane == 0) mbar_arrive(bar);
        } else if (lane == 0) {
          mbar_arrive_expect_tx(bar, Q_BYTES);
          for (int c = 0; c < 2; ++c)
            tma_load_3d(base + OFF_Q + c * QB * 128, &rq.tq, bar, c * 64, qb * QB, bh);
        }
      }
      ok = stream_item<GATHER, PERM>(rq, bh, begin, n, layout, ns, &rq.tk, rq.kg, base + OFF_K,
                                     ctrl.k_full, ctrl.k_empty, kc, 2, lane, wait);
    }
    cp_async_wait_all();
    if (*abort_flag) {
      // let issued copies land before the CTA exits (the last slots of the ring)
      volatile int32_t dummy = 0;
      for (int s = 0; s < KS; ++s)
        if (kc[s]) mbar_wait(smem_u32(&ctrl.k_full[s]), (kc[s] - 1) & 1, &dummy, p.err);
      if (qc) mbar_wait(smem_u32(&ctrl.q_full), (qc - 1) & 1, &dummy, p.err);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- V producer
    uint32_t vc[2] = {0u, 0u}, seq = 0;
    bool ok = true;
    while (ok) {
      const int slot = seq & 1;
      if (!wait(smem_u32(&ctrl.item_full[slot]), (seq >> 1) & 1, 18)) break;
      const int32_t it = ctrl.item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl.item_empty[slot]));
      ++seq;
      if (it < 0) break;
      const ReqParams& rq = p.req[fwd::req_of(p, it)];
      const int32_t li = it - rq.item_begin;
      const int4 i0 = __ldg(&rq.items[2 * li]);
      const int4 i1 = __ldg(&rq.items[2 * li + 1]);
      const int32_t bh = i0.x, begin = i0.z, n = i0.w - i0.z, layout = i1.x;
      const int32_t ns = (n + 1) >> 1;
      ok = stream_item<GATHER, PERM>(rq, bh, begin, n, layout, ns, &rq.tv, rq.vg, base + OFF_V,
                                     ctrl.v_full, ctrl.v_empty, vc, 3, lane, wait);
    }
    cp_async_wait_all();
    if (*abort_flag) {
      volatile int32_t dummy = 0;
      for (int s = 0; s < VS; ++s)
        if (vc[s]) mbar_wait(smem_u32(&ctrl.v_full[s]), (vc[s] - 1) & 1, &dummy, p.err);
    }
  } else if (warp == 1 || warp == 11) {
    // ------------------------------------------------ MMA issuers, one per group
    // Issuer g takes its group's steps of the item (item steps j = g, g + 2, ...;
    // group step t is item step 2 t + g) in the order QK(t), PV(t - 1): the PV of
    // group step t - 2 is issued before QK(t) reuses that step's S^T buffer.
    // Two issuing threads keep the tensor pipe fed while either one waits.
    if (lane == 0) {
      const int g = warp == 1 ? 0 : 1;
      uint32_t kc = 0, vc = 0, qc = 0, seq = 0, oc = 0;   // this group's K / V slot loads, items
      uint32_t gq = 0, gp = 0;                            // QKs / PVs issued for the group
      int64_t tiles = 0;
      bool ok = true;
      if (p.test_stall) ok = wait(smem_u32(&ctrl.never), 0, 4);
      while (ok) {
        const int slot = seq & 1;
        if (!wait(smem_u32(&ctrl.item_full[slot]), (seq >> 1) & 1, 5)) break;
        const int32_t it = ctrl.item_slot[slot];
        mbar_arrive(smem_u32(&ctrl.item_empty[slot]));
        ++seq;
        if (it < 0) break;
        const ReqParams& rq = p.req[fwd::req_of(p, it)];
        const int32_t li = it - rq.item_begin;
        const int4 i0 = __ldg(&rq.items[2 * li]);
        const int4 i1 = __ldg(&rq.items[2 * li + 1]);
        const int32_t n = i0.w - i0.z, ns = (n + 1) >> 1;
        if (g == 0) tiles += n;
        if (ns == 0) continue;
        const bool gath = GATHER || (PERM && i1.x != 0);
        const int32_t nt = (ns - g + 1) >> 1;             // this group's steps in the item
        if (!wait(smem_u32(&ctrl.q_full), qc & 1, 6)) break;
        ++qc;
        if (nt == 0) {
          // a one-step item leaves group 1 without work: it releases the query
          // tile and takes the item's O^T phases without MMAs
          mbar_arrive(smem_u32(&ctrl.q_empty));
          if (!wait(smem_u32(&ctrl.o_empty), (oc & 1) ^ 1, 10)) break;
          ++oc;
          mbar_arrive(smem_u32(&ctrl.o_full));
          continue;
        }
        if (gath) fence_proxy_async_smem();
        for (int32_t t = 0; t <= nt && ok; ++t) {
          if (t < nt) {
            // S^T = K Q^T for group step t (K slot g)
            if (!wait(smem_u32(&ctrl.k_full[g]), kc & 1, 7)) { ok = false; break; }
            ++kc;
            if (gath) fence_proxy_async_smem();
            tc_fence_after();
            const uint32_t sK = base + OFF_K + g * KV_BYTES;
            const uint32_t sb = gq & 1;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t a = sdesc_sw128(sK + (kk >> 2) * (2 * KT * 128) + (kk & 3) * 32, 16, 1024);
              const uint64_t b = sdesc_sw128(base + OFF_Q + (kk >> 2) * (QB * 128) + (kk & 3) * 32, 16, 1024);
              mma_bf16_ss(tmem + g * TM_GROUP + sb * QB, a, b, IDESC_QK, kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&ctrl.s_full[g][sb]));
            mma_commit(smem_u32(&ctrl.k_empty[g]));
            if (t == nt - 1) mma_commit(smem_u32(&ctrl.q_empty));
            ++gq;
          }
          if (t >= 1) {
            // O^T += V^T P^T for group step t - 1 (V slot g)
            const int32_t tt = t - 1;
            const uint32_t pb = gp & 1;                   // the group's P^T buffer of this step
            if (!wait(smem_u32(&ctrl.p_full[g][pb]), (gp >> 1) & 1, 8)) { ok = false; break; }
            if (!wait(smem_u32(&ctrl.v_full[g]), vc & 1, 9)) { ok = false; break; }
            ++vc;
            if (gath) fence_proxy_async_smem();
            if (tt == 0) {
              // the previous item's epilogue has read both groups' O^T
              if (!wait(smem_u32(&ctrl.o_empty), (oc & 1) ^ 1, 10)) { ok = false; break; }
              ++oc;
            }
            tc_fence_after();
            const uint32_t sV = base + OFF_V + g * KV_BYTES;
            const uint32_t sP = base + OFF_P + (2 * g + pb) * P_BYTES;
#pragma unroll
            for (int kk = 0; kk < (2 * KT) / 16; ++kk) {
              const uint64_t a = sdesc_sw128(sV + kk * 16 * 128, 2 * KT * 128, 1024);
              const uint64_t b = sdesc_sw128(sP + kk * 16 * 128, 2 * KT * 128, 1024);
              mma_bf16_ss(tmem + g * TM_GROUP + TM_O, a, b, IDESC_PV, (tt > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(smem_u32(&ctrl.v_empty[g]));
            mma_commit(smem_u32(&ctrl.pv_done[g][pb]));
            if (tt == nt - 1) mma_commit(smem_u32(&ctrl.o_full));
            ++gp;
          }
        }
      }
      if (p.tiles_done && tiles) atomicAdd(p.tiles_done, static_cast<unsigned long long>(tiles));
      mma_commit(smem_u32(&ctrl.final_bar[g]));
      volatile int32_t dummy = 0;
      mbar_wait(smem_u32(&ctrl.final_bar[g]), 0, &dummy, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- softmax groups
    const int g = (warp - 3) >> 2;                       // 0: warps 3..6, 1: warps 7..10
    const int quad = warp & 3;                           // TMEM lane quarter
    const int r = quad * 32 + lane;                      // key lane of S^T; d row of O^T
    const int half = r >> 6, c = r & 63;                 // the step's tile and key in it
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tg = tmem + lane_off + g * TM_GROUP;
    const uint32_t tl = tmem + lane_off + TM_L + g * QB; // this key's row-sum shares
    uint8_t* stage = smem_gen + OFF_P;                   // epilogue: O of the item, 64 x 256 B
    uint32_t seq = 0, gs = 0, grp_cnt = 0, pair_cnt = 0, o_seq = 0;
    bool ok = true;
    // barriers of the group's four warps / of both groups, bounded like every wait
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl.grp[g]));
      const bool r2 = wait(smem_u32(&ctrl.grp[g]), grp_cnt & 1, 11);
      ++grp_cnt;
      return r2;
    };
    auto pair_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl.pair));
      const bool r2 = wait(smem_u32(&ctrl.pair), pair_cnt & 1, 12);
      ++pair_cnt;
      return r2;
    };
    while (ok) {
      const int slot = seq & 1;
      if (!wait(smem_u32(&ctrl.item_full[slot]), (seq >> 1) & 1, 13)) break;
      const int32_t it = ctrl.item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl.item_empty[slot]));
      ++seq;
      if (it < 0) break;
      const ReqParams& rq = p.req[fwd::req_of(p, it)];
      const int32_t li = it - rq.item_begin;
      const int4 i0 = __ldg(&rq.items[2 * li]);
      const int4 i1 = __ldg(&rq.items[2 * li + 1]);
      const int32_t bh = i0.x, qb = i0.y, begin = i0.z, n = i0.w - i0.z, layout = i1.x;
      const int32_t ns = (n + 1) >> 1;
      const int32_t q0 = qb * QB;
      // entry and descriptor of this thread's tile in step `step`
      auto fetch = [&](int32_t step, int32_t& kv, int32_t& desc, uint4& d0, uint4& d1, bool& has) {
        const int32_t e = begin + 2 * step + half;
        has = e < begin + n;
        kv = 0;
        desc = -1;
        d0 = make_uint4(0u, 0u, 0u, 0u);
        d1 = d0;
        if (has) {
          const int2 en = __ldg(&rq.entries[e]);
          kv = en.x;
          desc = en.y;
          if (desc >= 0) {
            d0 = __ldg(&rq.descs[2 * desc]);
            d1 = __ldg(&rq.descs[2 * desc + 1]);
          }
        }
      };
      for (int32_t j = g; j < ns; j += 2) {
        const uint32_t t = gs;                           // this group's step count
        const uint32_t sb = t & 1;
        const bool first = j == g;                       // the group's first step of the item
        // this thread's tile: fetched before the wait for the step's S^T, which
        // hides the load latency
        int32_t kv, desc;
        uint4 d0, d1;
        bool has;
        fetch(j, kv, desc, d0, d1, has);
        // Queries this key may see: 64 bits (w0: queries 0..31, w1: 32..63).
        uint32_t w0 = 0xFFFFFFFFu, w1 = 0xFFFFFFFFu;
        if (!has) {
          w0 = w1 = 0u;                                   // no second tile in this step
        } else if (desc >= 0) {
          if (GATHER) {
            // list form: the key slot is listed for the whole block, or padding
            const uint32_t cw = (c < 32) ? d0.x : d0.y;
            if (!((cw >> (c & 31)) & 1u)) w0 = w1 = 0u;
          } else if ((d0.x & 0xFF) == 0) {
            // band form (temporal-major SVG heads): queries whose F-token
            // segment is within R of this key's
            // (N < 2^24, so the key and its segment fit 32-bit division; the
            // interval bounds are formed in 64 bits)
            const int32_t Fb = static_cast<int32_t>(d1.w);
            const int64_t Rb = d1.z;
            const int32_t k = kv + c;
            w0 = w1 = 0u;
            if (k < rq.N) {
              const int64_t seg = k / Fb;
              const int64_t lo_a = (seg - Rb) * Fb - q0, hi_a = (seg + Rb + 1) * Fb - q0;
              const int64_t hi_n = static_cast<int64_t>(rq.N) - q0;
              const int lo = static_cast<int>(lo_a > 0 ? lo_a : 0);
              const int64_t hcap = hi_a < hi_n ? hi_a : hi_n;
              const int hi = static_cast<int>(hcap < QB ? (hcap > 0 ? hcap : 0) : QB);
              if (lo < hi) range64(w0, w1, lo, hi);
            }
          } else {
            // grid form: this key's column segment, then the allowed row segments
            const int n_r = d0.x & 0xFF, n_c = (d0.x >> 8) & 0xFF;
            const int c_end = static_cast<int>(dbyte(d0, d1, 10 + n_c));
            w0 = w1 = 0u;
            if (c < c_end) {
              int cs = 0;
#pragma unroll
              for (int k = 1; k < 8; ++k)
                if (k < n_c && static_cast<int>(dbyte(d0, d1, 10 + k)) <= c) cs = k;
              const uint64_t bits = (static_cast<uint64_t>(d1.w) << 32) | d1.z;
#pragma unroll
              for (int rr = 0; rr < 8; ++rr) {
                if (rr < n_r && ((bits >> (rr * 8 + cs)) & 1ull)) {
                  const int lo = static_cast<int>(dbyte(d0, d1, 2 + rr));
                  const int hi = (rr + 1 < n_r) ? static_cast<int>(dbyte(d0, d1, 3 + rr)) : QB;
                  range64(w0, w1, lo, hi);
                }
              }
            }
          }
        }
        if (!wait(smem_u32(&ctrl.s_full[g][sb]), (t >> 1) & 1, 14)) { ok = false; break; }
        tc_fence_after();
        // One half (32 queries) of this key's logits from TMEM, masked, as
        // y = x * scale (base 2).
        auto load_y = [&](int h, float (&y)[32]) {
          uint32_t rr[32];
          tmem_ld32(tg + sb * QB + 32 * h, rr);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            fwd::fma2(y[i], y[i + 1], __uint_as_float(rr[i]), __uint_as_float(rr[i + 1]), p.scale_log2, 0.f);
          const uint32_t w = h ? w1 : w0;
          if (w != 0xFFFFFFFFu) {                         // not every query of this key allowed
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (!((w >> i) & 1u)) y[i] = -INFINITY;
          }
        };
        // P = 2^(y - m) of one half against the reference m (shared memory);
        // returns the largest y - m
        auto exp_half = [&](float (&y)[32], const float* m) -> float {
          float tm = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(m + i);
            const float d0 = y[i] - m4.x, d1 = y[i + 1] - m4.y, d2 = y[i + 2] - m4.z, d3 = y[i + 3] - m4.w;
            tm = fwd::max3f(tm, d0, d1);
            tm = fwd::max3f(tm, d2, d3);
            y[i] = ex2_approx(d0);
            y[i + 1] = ex2_approx(d1);
            y[i + 2] = ex2_approx(d2);
            y[i + 3] = ex2_approx(d3);
          }
          return tm;
        };
        // The optimistic pass works on the raw logits: P = 2^(x * scale - m) with
        // the scale and the reference in one FFMA per element (masked: -inf);
        // returns the largest x * scale - m.  No clamp: a half whose largest
        // exponent is above the threshold takes the correction, which rewrites
        // its P^T and never uses its optimistic values
        auto load_x = [&](int h, float (&x)[32]) {
          uint32_t rr[32];
          tmem_ld32(tg + sb * QB + 32 * h, rr);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(rr[i]);
          const uint32_t w = h ? w1 : w0;
          if (w != 0xFFFFFFFFu) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (!((w >> i) & 1u)) x[i] = -INFINITY;
          }
        };
        auto exp_half_x = [&](float (&x)[32], const float* m) -> float {
          float tm = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(m + i);
            float d0, d1, d2, d3;
            fma2c(d0, d1, x[i], x[i + 1], p.scale_log2, -m4.x, -m4.y);
            fma2c(d2, d3, x[i + 2], x[i + 3], p.scale_log2, -m4.z, -m4.w);
            tm = fwd::max3f(tm, d0, d1);
            tm = fwd::max3f(tm, d2, d3);
            x[i] = ex2_approx(d0);
            x[i + 1] = ex2_approx(d1);
            x[i + 2] = ex2_approx(d2);
            x[i + 3] = ex2_approx(d3);
          }
          return tm;
        };
        // this step's P^T buffer (t & 1) is free once the group's PV two steps
        // back has read it (across items too: then it has long completed)
        if (t >= 2) {
          if (!wait(smem_u32(&ctrl.pv_done[g][sb]), ((t - 2) >> 1) & 1, 16)) { ok = false; break; }
        }
        uint8_t* prow = smem_gen + OFF_P + (2 * g + sb) * P_BYTES + r * 128;
        auto store_p = [&](int h, const float (&pv)[32]) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int uu = 4 * h + u;
            const float* pp = pv + 8 * u;
            *reinterpret_cast<uint4*>(prow + ((uu ^ (r & 7)) << 4)) =
                make_uint4(pack_bf16x2(pp[0], pp[1]), pack_bf16x2(pp[2], pp[3]),
                           pack_bf16x2(pp[4], pp[5]), pack_bf16x2(pp[6], pp[7]));
          }
        };
        // exact column maximum of this step over the group's 128 keys, raised
        // into the reference (mold keeps the previous one, alpha the factor)
        auto raise_reference = [&]() -> bool {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            float y[32];
            load_y(h, y);
            warp_reduce<true, 32>(y, lane);
            ctrl.red[g][quad][32 * h + lane] = y[0];
          }
          if (!group_sync()) return false;
          if (r < QB) {
            const float mo = ctrl.mref[g][r];
            const float mt = fmaxf(fmaxf(ctrl.red[g][0][r], ctrl.red[g][1][r]),
                                   fmaxf(ctrl.red[g][2][r], ctrl.red[g][3][r]));
            const float mn = fmaxf(mo, mt);
            ctrl.mold[g][r] = mo;
            ctrl.alpha[g][r] = ex2_approx(mo - mn);
            ctrl.mref[g][r] = mn;
          }
          return group_sync();
        };
        if (first) {
          // the item's first step for this group: the reference is taken from
          // the step itself, then P and the row-sum shares
          if (!raise_reference()) { ok = false; break; }
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            float y[32];
            load_y(h, y);
            exp_half(y, ctrl.mref[g] + 32 * h);
            store_p(h, y);
            uint32_t rl[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) rl[i] = __float_as_uint(y[i]);
            tmem_st32(tl + 32 * h, rl);
          }
        } else {
          // optimistic pass against the current reference; the group then
          // checks that no logit exceeded it by more than the threshold.  A
          // warp adds a half's P to its row-sum shares only when no exponent
          // of that half is above the threshold (`added`, warp-uniform)
          float tmax = -INFINITY;
          uint32_t added = 0u;
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            float y[32];
            uint32_t rl[32];
            load_x(h, y);
            tmem_ld32(tl + 32 * h, rl);
            const float th = exp_half_x(y, ctrl.mref[g] + 32 * h);
            tmax = fmaxf(tmax, th);
            store_p(h, y);
            tc_wait_ld();
            if (!__any_sync(0xFFFFFFFFu, th > kFixThreshold)) {
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float a = __uint_as_float(rl[i]), b = __uint_as_float(rl[i + 1]);
                fwd::add2(a, b, y[i], y[i + 1]);
                rl[i] = __float_as_uint(a);
                rl[i + 1] = __float_as_uint(b);
              }
              tmem_st32(tl + 32 * h, rl);
              added |= 1u << h;
            }
          }
          if (__any_sync(0xFFFFFFFFu, tmax > kFixThreshold) && lane == 0)
            ctrl.fixflag[g][t & 1] = static_cast<int32_t>(t);
          if (!group_sync()) { ok = false; break; }
          if (ctrl.fixflag[g][t & 1] == static_cast<int32_t>(t)) {
            // correction: raise the reference to the step's exact maximum,
            // replace this step's optimistic shares (l = (l - p_old) a + p_new
            // for the halves that added them, l a + p_new for the others),
            // rewrite P^T, and rescale O^T once the group's previous PV is done
            tc_wait_st();
            if (!raise_reference()) { ok = false; break; }
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              float y[32], yo[32];
              uint32_t rl[32];
              load_x(h, y);
#pragma unroll
              for (int i = 0; i < 32; ++i) yo[i] = y[i];
              tmem_ld32(tl + 32 * h, rl);
              exp_half_x(yo, ctrl.mold[g] + 32 * h);          // the optimistic P, as added
              exp_half_x(y, ctrl.mref[g] + 32 * h);
              store_p(h, y);
              tc_wait_ld();
              const bool was_added = (added >> h) & 1u;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float a = ctrl.alpha[g][32 * h + i];
                const float lo = __uint_as_float(rl[i]);
                rl[i] = __float_as_uint((was_added ? lo - yo[i] : lo) * a + y[i]);
              }
              tmem_st32(tl + 32 * h, rl);
            }
            if (!wait(smem_u32(&ctrl.pv_done[g][(t - 1) & 1]), ((t - 1) >> 1) & 1, 15)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int blk = 0; blk < 2; ++blk) {
              uint32_t rr[32];
              tmem_ld32(tg + TM_O + 32 * blk, rr);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                rr[i] = __float_as_uint(__uint_as_float(rr[i]) * ctrl.alpha[g][32 * blk + i]);
              tmem_st32(tg + TM_O + 32 * blk, rr);
            }
          }
        }
        tc_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl.p_full[g][sb]));
        ++gs;
      }
      if (!ok) break;
      // ----------------------------------------------------------- epilogue
      // this group's row sums: its keys' shares summed over the 128 lanes
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[32];
        if (ns > g) {
          uint32_t rl[32];
          tmem_ld32(tl + 32 * h, rl);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(rl[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        warp_reduce<false, 32>(v, lane);
        ctrl.red[g][quad][32 * h + lane] = v[0];
      }
      if (!group_sync()) break;
      if (r < QB)
        ctrl.lsum[g][r] = (ctrl.red[g][0][r] + ctrl.red[g][1][r]) + (ctrl.red[g][2][r] + ctrl.red[g][3][r]);
      if (!pair_sync()) break;
      // merge the two groups' halves of the item (per query)
      if (g == 0 && r < QB) {
        const float m0 = ctrl.mref[0][r], m1 = ctrl.mref[1][r];
        const float l0 = ctrl.lsum[0][r], l1 = ctrl.lsum[1][r];
        const float m = fmaxf(m0, m1);
        const float a0 = l0 > 0.f ? ex2_approx(m0 - m) : 0.f;
        const float a1 = l1 > 0.f ? ex2_approx(m1 - m) : 0.f;
        const float l = a0 * l0 + a1 * l1;
        const float inv = l > 0.f ? __fdividef(1.f, l) : 0.f;
        ctrl.fac[0][r] = a0 * inv;
        ctrl.fac[1][r] = a1 * inv;
        ctrl.lse2[r] = l > 0.f ? m + __log2f(l) : -INFINITY;
      }
      if (!pair_sync()) break;
      if (r < QB) ctrl.mref[g][r] = kMrefInit;          // for the next item
      // split-KV unit (part i1.w of the i1.z parts of work item i1.y): the
      // normalised partial O (fp32, [q][d]) and lse (base 2) go to the plan's
      // workspace instead of the output, and the last part to finish merges
      const bool split = i1.z > 1;
      const int64_t unit = split ? static_cast<int64_t>(i1.y) * i1.z + i1.w : 0;
      float* const part = split ? rq.part_o + unit * QB * D : nullptr;
      if (split && ns == 0) {
        for (int q = 32 * g; q < 32 * g + 32; ++q) part[q * D + r] = 0.f;
      }
      if (ns > 0) {
        // O = fac0 O0 + fac1 O1 for queries [32 g, 32 g + 32), transposed into
        // the staging tile: element (q, d) at row q (256 B), 16-byte unit
        // (d / 8) ^ (q & 7), byte 2 (d % 8)
        if (!wait(smem_u32(&ctrl.o_full), o_seq & 1, 17)) break;
        ++o_seq;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 32 * g; c0 < 32 * g + 32; c0 += 16) {
          uint32_t ra[16], rb[16];
          tmem_ld16(tmem + lane_off + TM_O + c0, ra);
          if (ns > 1) tmem_ld16(tmem + lane_off + TM_GROUP + TM_O + c0, rb);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int q = c0 + i;
            float o = __uint_as_float(ra[i]) * ctrl.fac[0][q];
            if (ns > 1) o += __uint_as_float(rb[i]) * ctrl.fac[1][q];
            if (split)
              part[q * D + r] = o;
            else
              *reinterpret_cast<__nv_bfloat16*>(stage + q * 256 + (((r >> 3) ^ (q & 7)) << 4) + (r & 7) * 2) =
                  __float2bfloat16_rn(o);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl.o_empty));
      }
      if (!pair_sync()) break;
      if (split) {
        if (g == 0 && r < QB) rq.part_lse[unit * QB + r] = ctrl.lse2[r];
        __threadfence();
        if (!pair_sync()) break;
        if (g == 0 && r == 0) ctrl.split_last = (atomicAdd(rq.part_cnt + i1.y, 1) == i1.z - 1) ? 1 : 0;
        if (!pair_sync()) break;
        if (ctrl.split_last) {
          // merge the parts: 256 threads, row q, quarter qt (32 d values)
          __threadfence();
          const int t8 = g * 128 + r, q = t8 & 63, qt = t8 >> 6;
          const int32_t tq = q0 + q;
          if (tq < rq.N) {
            const int64_t u0 = static_cast<int64_t>(i1.y) * i1.z;
            float w[4], M = -INFINITY;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              w[k] = (k < i1.z) ? __ldcg(rq.part_lse + (u0 + k) * QB + q) : -INFINITY;
              M = fmaxf(M, w[k]);
            }
            float L = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              w[k] = (M == -INFINITY) ? 0.f : ex2_approx(w[k] - M);   // ex2(-inf) = 0
              L += w[k];
            }
            const float inv = (L > 0.f) ? __fdividef(1.f, L) : 0.f;
            const int32_t orow = (PERM && layout) ? unpermute(tq, rq.F, rq.S) : tq;
            uint4* dst = reinterpret_cast<uint4*>(rq.out + (static_cast<size_t>(bh) * rq.N + orow) * D + qt * 32);
            // every part's two float4 of a chunk are loaded together (parts past
            // i1.z load nothing and weigh 0), two chunks in flight
            const float4* src[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              src[k] = reinterpret_cast<const float4*>(rq.part_o + ((u0 + (k < i1.z ? k : 0)) * QB + q) * D + qt * 32);
#pragma unroll 2
            for (int u = 0; u < 4; ++u) {
              float4 x[4][2];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const bool on = k < i1.z;
                x[k][0] = on ? __ldcg(src[k] + 2 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
                x[k][1] = on ? __ldcg(src[k] + 2 * u + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
              }
              float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float wk = w[k] * inv;
                acc[0] += wk * x[k][0].x; acc[1] += wk * x[k][0].y; acc[2] += wk * x[k][0].z; acc[3] += wk * x[k][0].w;
                acc[4] += wk * x[k][1].x; acc[5] += wk * x[k][1].y; acc[6] += wk * x[k][1].z; acc[7] += wk * x[k][1].w;
              }
              dst[u] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                  pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
            }
            if (qt == 0) rq.lse[static_cast<size_t>(bh) * rq.N + orow] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
          }
        }
      } else {
        // 256 threads store the 64 rows: row q, quarter qt (32 d values, 64 B)
        const int t8 = g * 128 + r, q = t8 & 63, qt = t8 >> 6;
        const int32_t tq = q0 + q;
        if (tq < rq.N) {
          const int32_t orow = (PERM && layout) ? unpermute(tq, rq.F, rq.S) : tq;
          uint4* dst = reinterpret_cast<uint4*>(rq.out + (static_cast<size_t>(bh) * rq.N + orow) * D + qt * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
            if (ns > 0) v4 = *reinterpret_cast<const uint4*>(stage + q * 256 + (((qt * 4 + u) ^ (q & 7)) << 4));
            dst[u] = v4;
          }
          if (qt == 0) {
            const float l2 = ctrl.lse2[q];
            rq.lse[static_cast<size_t>(bh) * rq.N + orow] = (l2 > -INFINITY) ? l2 * kLn2 : -INFINITY;
          }
        }
      }
      // the staging tile is free and the reset maxima are visible to both groups
      if (!pair_sync()) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int MODE, int MAXR>
tsr_status launch_t(const FwdParamsT<MAXR>& prm, int n_items, int device, cudaStream_t stream) {
  auto kern = bsa_fwd_t_kernel<MODE, MAXR>;
  static bool attr_set[64] = {false};
  if (device < 0 || device >= 64 || !attr_set[device]) {
    TSR_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    if (device >= 0 && device < 64) attr_set[device] = true;
  }
  const int grid = std::min(n_items, num_sms(device));
  if (grid <= 0) return TSR_OK;
  kern<<<grid, kThreads, SMEM_BYTES, stream>>>(prm);
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

tsr_status launch_t_mode(const fwd::FwdParams& prm, int mode, int n_items, int device,
                         cudaStream_t stream);
tsr_status launch_t_mode(const fwd::FwdParamsBatch& prm, int mode, int n_items, int device,
                         cudaStream_t stream);

}  // namespace fwd_t
}  // namespace tsr
