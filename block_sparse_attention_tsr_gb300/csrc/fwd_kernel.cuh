// fwd_kernel.cuh -- the block-sparse attention forward kernel on tcgen05 tensor
// cores, shared by the per-mode translation units (fwd_tma.cu, fwd_perm.cu,
// fwd_list.cu); the host side is in fwd.cu.
//
// One persistent CTA per SM slot pulls work items (one 128-row query tile plus
// its list of physical K/V tiles, longest first) from an atomic counter.  Inside
// a CTA three roles run concurrently and hand data over through mbarriers:
//
//   warp 0      producer: the query tile once per item, then the K and V tiles
//               of the item's list through a STAGES-deep shared-memory ring, by
//               TMA, or by row gathers for key lists and temporal-major items.
//               Empty tiles are not in the list, so they are never loaded
//               (Splash digest, "Splash Attention": empty tiles are bypassed).
//   warp 1      MMA issuer (one thread): S = Q K^T into TMEM (double buffered),
//               then O += P V with P read from TMEM; QK of tile j+1 is issued
//               before PV of tile j so the tensor pipe stays busy while the
//               softmax of tile j runs.
//   warps 2..5  softmax, one query row per thread (TMEM lane = row): scale,
//               element mask on boundary tiles only (Splash digest: exact
//               coordinate masking limited to boundary tiles), online softmax in
//               fp32 with lazy rescaling, P to TMEM as bf16, and the epilogue
//               O / l -> bf16, lse = m + ln l.  Rows that see no allowed key get
//               O = 0 and lse = -inf.
//
// The arithmetic is the masked softmax attention of the Tessera abstract (block-
// sparse attention over the logical mask, every named interaction kept); the
// online (streaming) softmax is the standard one-pass rewrite of it.
#pragma once
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace tsr {
namespace fwd {


// Kernel modes: which loads an item may take.
//   kModeTma   every tile by TMA (UNIFORM, SEGMENTS, and SVG plans without
//              temporal heads)
//   kModePerm  TMA, or row gathers through the inverse temporal-major
//              permutation for the items of temporal heads (SVG)
//   kModeList  K / V rows gathered from a key list (KEYLIST)
enum : int { kModeTma = 0, kModePerm = 1, kModeList = 2 };

// One attention request: its tensors and its tile plan.  A launch covers one
// request (tsr_bsa_forward) or up to kMaxBatch requests of possibly different
// shapes (tsr_bsa_forward_batch); their work items are numbered one after the
// other, request r's from req[r].item_begin.
constexpr int kMaxBatch = 16;

struct ReqParams {
  CUtensorMap tq, tk, tv;        // caller layout, 3-D {d, N, B*H}
  const int4* items;             // tsr_plan_item, 2 x int4 each
  const int2* entries;
  const uint4* descs;            // 32 B each
  __nv_bfloat16* out;
  float* lse;
  // rows loaded by index: KEYLIST keys named by gidx, and every row of a
  // temporal-major (SVG temporal) item
  const __nv_bfloat16* qg;
  const __nv_bfloat16* kg;
  const __nv_bfloat16* vg;
  const int32_t* gidx;
  // split-KV plans: each unit's partial O (fp32 [bm][d]) and lse (base 2, [bm])
  // by unit index, one arrival counter per work item (zeroed before the launch)
  float* part_o;
  float* part_lse;
  int32_t* part_cnt;
  int32_t item_begin, N, F, S, slice_m;
};

// Launch parameters for up to MAXR requests: MAXR = 1 for tsr_bsa_forward
// (the request index is then a constant), kMaxBatch for batched launches.
template <int MAXR>
struct FwdParamsT {
  int32_t* counter;
  uint32_t* err;
  unsigned long long* tiles_done;   // debug checks: tiles computed, else null
  int32_t n_items;               // over all requests
  int32_t n_req;
  float scale_log2;              // log2(e) / sqrt(d)
  int32_t test_stall;           // test only: the MMA issuer waits on a barrier nobody signals
  uint64_t timeout_ns;          // bound of every wait
  ReqParams req[MAXR];
};
using FwdParams = FwdParamsT<1>;
using FwdParamsBatch = FwdParamsT<kMaxBatch>;

// The request holding work item `it` (requests are few: a linear scan).
template <int MAXR>
__device__ __forceinline__ int req_of(const FwdParamsT<MAXR>& p, int32_t it) {
  if constexpr (MAXR == 1) {
    return 0;
  } else {
    int r = 0;
    for (int i = 1; i < p.n_req; ++i)
      if (it >= p.req[i].item_begin) r = i;
    return r;
  }
}

// Rescale the running output only when the running maximum grew by more than
// this many powers of two: P = 2^(x - m_ref) then stays below 2^8, far inside
// bf16 and fp32 range, and O / l is unchanged because O and l share the factor.
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

struct alignas(8) Ctrl {
  uint64_t q_full, q_empty;
  uint64_t k_full[8], v_full[8], k_empty[8], v_empty[8];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, o_full, o_empty;
  uint64_t item_full[2], item_empty[2];
  uint64_t final_bar, never;
  uint64_t split_bar;          // split-KV epilogue: the four softmax warps
  int32_t item_slot[2];
  int32_t split_last;          // this CTA's unit was the last part of its item
  uint32_t tmem_base;
  int32_t abort_flag;
};

template <int D, int BN, int STAGES, int CTAS>
struct Cfg {
  static constexpr int BM = kBM;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int SMEM = Q_BYTES + 2 * STAGES * KV_BYTES + 1024;
  // TMEM per CTA (512 columns per SM shared by CTAS CTAs) holds two BN-column S
  // buffers (P is written over S as bf16), O (D columns) and, where the rest
  // leaves room, the query tile (D / 2 columns of bf16 pairs).  With Q in TMEM
  // the S = Q K^T MMAs read A from TMEM and shared memory feeds the tensor core
  // only K and V (measured: +6 to +9 % on one-CTA variants).  Two-CTA variants
  // at d = 128 have no room for it; giving up the second S buffer to make room
  // was measured 25 % slower, because QK of tile j+1 then waits for the softmax
  // of tile j.
  static constexpr int BUDGET = 512 / CTAS;
  static constexpr bool Q_TMEM = 2 * BN + D + D / 2 <= BUDGET;
  static constexpr int O_COL = 2 * BN;
  static constexpr int Q_COL = O_COL + D;
  static constexpr int COLS = O_COL + D + (Q_TMEM ? D / 2 : 0);
  static constexpr int TMEM_COLS = COLS <= 128 ? 128 : COLS <= 256 ? 256 : 512;
  static_assert(TMEM_COLS * CTAS <= 512, "TMEM");
  static constexpr uint32_t IDESC_QK = idesc_bf16(128, BN, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
  static_assert(STAGES >= 2 && STAGES <= 8, "stages");
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(BN == 64 || BN == 128, "kv tile");
};

__device__ __forceinline__ int32_t unpermute(int32_t tp, int32_t F, int32_t S) {
  return (tp % F) * S + tp / F;
}

// Byte i of a 32-byte descriptor held in two uint4 registers (selects, no
// local-memory indexing when i is not a compile-time constant).
__device__ __forceinline__ uint32_t desc_byte(const uint4& a, const uint4& b, int i) {
  const int w = i >> 2;
  const uint32_t lo = (w & 1) ? ((w & 2) ? a.w : a.y) : ((w & 2) ? a.z : a.x);
  const uint32_t hi = (w & 1) ? ((w & 2) ? b.w : b.y) : ((w & 2) ? b.z : b.x);
  return (((w & 4) ? hi : lo) >> ((i & 3) * 8)) & 0xFFu;
}

// Packed fp32 pair arithmetic (two lanes per instruction).
__device__ __forceinline__ void fma2(float& y0, float& y1, float x0, float x1, float s, float b) {
  asm("{\n\t.reg .b64 xa, sa, ba;\n\tmov.b64 xa, {%2, %3};\n\tmov.b64 sa, {%4, %4};\n\t"
      "mov.b64 ba, {%5, %5};\n\tfma.rn.f32x2 xa, xa, sa, ba;\n\tmov.b64 {%0, %1}, xa;\n\t}"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(s), "f"(b));
}
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb;\n\tmov.b64 ra, {%0, %1};\n\tmov.b64 rb, {%2, %3};\n\t"
      "add.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Columns [lo, hi) of a BN-bit mask, added to words[].
template <int BN>
__device__ __forceinline__ void add_range(uint32_t (&words)[BN / 32], int lo, int hi) {
#pragma unroll
  for (int w = 0; w < BN / 32; ++w) {
    const int a = max(lo - 32 * w, 0), b = min(hi - 32 * w, 32);
    if (a < b) {
      const uint32_t hi_mask = (b == 32) ? 0xFFFFFFFFu : ((1u << b) - 1u);
      words[w] |= hi_mask & ~((1u << a) - 1u);
    }
  }
}

// Copy ROWS rows of d bf16 values, row r from source row rows[r / 32] of lane
// r % 32 of a head, into a tile in the 128-byte swizzled K-major layout
// (64-element chunks of ROWS rows), with 16-byte cp.async.  Completion on `bar`:
//   LANE_ARRIVALS  each lane arrives once its own copies have landed (the
//                  barrier expects 32 arrivals; key-list tiles, all gathered)
//   otherwise      each lane ties its copies to the current phase and lane 0
//                  gives the phase its single ordinary arrival (the barrier
//                  expects one, so TMA and gathered tiles can share it)
template <int D, int ROWS, bool LANE_ARRIVALS>
__device__ __forceinline__ void gather_tile(const __nv_bfloat16* head_base,
                                            const int32_t (&rows)[ROWS / 32], uint32_t dst,
                                            uint32_t bar, int lane) {
  constexpr int UNITS = D / 8;        // 16-byte units per row
  constexpr int RPI = 32 / UNITS;     // rows per warp instruction
#pragma unroll
  for (int m = 0; m < ROWS / RPI; ++m) {
    const int row = RPI * m + lane / UNITS;
    const int src = __shfl_sync(0xFFFFFFFFu, rows[(RPI * m) / 32], row & 31);
    const int j = lane % UNITS, c = j >> 3, u = j & 7;
    const void* g = reinterpret_cast<const uint8_t*>(head_base + static_cast<size_t>(src) * D) + j * 16;
    cp_async_16(dst + c * ROWS * 128 + row * 128 + ((u ^ (row & 7)) << 4), g);
  }
  if constexpr (LANE_ARRIVALS) {
    cp_async_arrive_noinc(bar);
  } else {
    cp_async_arrive(bar);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  }
}

template <int D, int BN, int STAGES, int CTAS, int MODE, int MAXR>
__global__ void __launch_bounds__(192, CTAS) bsa_fwd_kernel(const __grid_constant__ FwdParamsT<MAXR> p) {
  using C = Cfg<D, BN, STAGES, CTAS>;
  constexpr bool GATHER = MODE == kModeList;   // K / V rows named by a key list
  constexpr bool PERM = MODE == kModePerm;     // items may be temporal-major
  extern __shared__ uint8_t smem_raw[];
  __shared__ Ctrl ctrl;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK0 = base + C::Q_BYTES;
  const uint32_t sV0 = sK0 + STAGES * C::KV_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int32_t* abort_flag = &ctrl.abort_flag;

  if (threadIdx.x == 0) {
    // full barriers take one arrival (lane 0's: with the byte count for a TMA
    // tile, after every lane has tied its copies to the phase for a gathered
    // one), except the K / V barriers of key-list plans: one per producer lane
    mbar_init(smem_u32(&ctrl.q_full), 1);
    mbar_init(smem_u32(&ctrl.q_empty), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctrl.k_full[s]), GATHER ? 32 : 1);
      mbar_init(smem_u32(&ctrl.v_full[s]), GATHER ? 32 : 1);
      mbar_init(smem_u32(&ctrl.k_empty[s]), 1);
      mbar_init(smem_u32(&ctrl.v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctrl.s_full[b]), 1);
      mbar_init(smem_u32(&ctrl.p_full[b]), 4);
      mbar_init(smem_u32(&ctrl.item_full[b]), 1);
      mbar_init(smem_u32(&ctrl.item_empty[b]), 5);
    }
    mbar_init(smem_u32(&ctrl.pv_done), 1);
    mbar_init(smem_u32(&ctrl.o_full), 1);
    mbar_init(smem_u32(&ctrl.o_empty), 4);
    mbar_init(smem_u32(&ctrl.split_bar), 4);
    mbar_init(smem_u32(&ctrl.final_bar), 1);
    mbar_init(smem_u32(&ctrl.never), 1);
    ctrl.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctrl.tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&p.req[0].tq);
      tma_prefetch_desc(&p.req[0].tk);
      tma_prefetch_desc(&p.req[0].tv);
    }
    uint32_t item_seq = 0, kv_cnt = 0, q_cnt = 0, k_iss = 0, v_iss = 0;
    bool ok = true;
    // Rows loaded by index (gather_tile): KEYLIST tiles (FG-Attn abstract: only
    // the listed keys of a query block are loaded, packed into dense tiles in
    // shared memory) and temporal-major items (Splash digest: tokens permuted to
    // temporal-major order -- here the permutation is applied while loading, so
    // no permuted copy of Q, K, V is ever written).  Everything else is TMA.
    auto tma_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, int32_t row0,
                        int32_t rows, uint32_t bytes, int32_t bh_) {
      if (lane == 0) {
        mbar_arrive_expect_tx(bar, bytes);
        for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * rows * 128, map, bar, c * 64, row0, bh_);
      }
    };
    auto wait_free = [&](uint32_t bar, uint32_t parity) -> bool {
      return mbar_wait(bar, parity, abort_flag, p.err, p.timeout_ns);
    };
    while (ok) {
      int32_t it = 0;
      if (lane == 0) it = atomicAdd(p.counter, 1);
      it = __shfl_sync(0xFFFFFFFFu, it, 0);
      const bool done = it >= p.n_items;
      const int slot = item_seq & 1;
      if (!mbar_wait(smem_u32(&ctrl.item_empty[slot]), ((item_seq >> 1) & 1) ^ 1, abort_flag, p.err, p.timeout_ns)) break;
      if (lane == 0) {
        ctrl.item_slot[slot] = done ? -1 : it;
        mbar_arrive(smem_u32(&ctrl.item_full[slot]));
      }
      ++item_seq;
      if (done) break;
      const ReqParams& rq = p.req[req_of(p, it)];
      const int32_t li = it - rq.item_begin;
      const int4 i0 = __ldg(&rq.items[2 * li]);
      const int4 i1 = __ldg(&rq.items[2 * li + 1]);
      const int32_t bh = i0.x, q_tile = i0.y, begin = i0.z, end = i0.w, layout = i1.x;
      if (end <= begin) continue;
      const size_t head_off = static_cast<size_t>(bh) * rq.N * D;
      const bool perm = PERM && layout != 0;
      // source row of a temporal-major row t' (rows past N read row 0; masked)
      auto perm_row = [&](int32_t tp) -> int32_t { return tp < rq.N ? unpermute(tp, rq.F, rq.S) : 0; };
      if (!wait_free(smem_u32(&ctrl.q_empty), (q_cnt & 1) ^ 1)) break;
      if (perm) {
        int32_t rows[C::BM / 32];
#pragma unroll
        for (int m = 0; m < C::BM / 32; ++m) rows[m] = perm_row(q_tile * C::BM + 32 * m + lane);
        gather_tile<D, C::BM, false>(rq.qg + head_off, rows, sQ, smem_u32(&ctrl.q_full), lane);
      } else {
        tma_tile(&rq.tq, sQ, smem_u32(&ctrl.q_full), q_tile * C::BM, C::BM, C::Q_BYTES, bh);
      }
      ++q_cnt;
      // Where tile e's rows come from: its first key row (TMA, temporal-major),
      // or its slice of gidx (key lists; gathered tile e owns gidx[e * BN, +BN)).
      // Key-list sources are fetched one tile ahead, so the gidx load latency
      // overlaps the stage wait (measured +21 %); the others are fetched after
      // the stage wait, separately for K and V (fetching them earlier, or
      // reusing K's for V, measured 2 % slower on SVG).
      auto tile_src = [&](int32_t e, int32_t (&rows)[BN / 32]) -> int32_t {
        if constexpr (GATHER) {
#pragma unroll
          for (int m = 0; m < BN / 32; ++m) rows[m] = __ldg(rq.gidx + e * BN + 32 * m + lane);
          return e * BN;
        } else {
          return __ldg(&rq.entries[e]).x;
        }
      };
      // one K or V tile into stage buffer dst
      auto load_kv = [&](const CUtensorMap* map, const __nv_bfloat16* base, int32_t kv,
                         const int32_t (&src_rows)[BN / 32], uint32_t dst, uint32_t bar) {
        if (GATHER) {
          gather_tile<D, BN, true>(base + head_off, src_rows, dst, bar, lane);
        } else if (perm) {
          int32_t rows[BN / 32];
#pragma unroll
          for (int m = 0; m < BN / 32; ++m) rows[m] = perm_row(kv + 32 * m + lane);
          gather_tile<D, BN, false>(base + head_off, rows, dst, bar, lane);
        } else {
          tma_tile(map, dst, bar, kv, BN, C::KV_BYTES, bh);
        }
      };
      // K runs one tile ahead of V: K of tile i is needed by QK(i), which the
      // MMA issuer runs before PV(i-1); a K stage is released by its QK, a V
      // stage by its PV, so the K stream never waits behind a PV.
      const int32_t n = end - begin;
      int32_t kv_k = 0, rows_k[BN / 32] = {}, kv_v = 0, rows_v[BN / 32] = {};
      if (GATHER && n > 0) kv_k = tile_src(begin, rows_k);
      for (int32_t i = 0; i <= n && ok; ++i) {
        int32_t kv_n = 0, rows_n[BN / 32] = {};
        if (GATHER && i + 1 < n) kv_n = tile_src(begin + i + 1, rows_n);
        if (i < n) {
          const uint32_t kvi = kv_cnt + i;
          const int s = kvi % STAGES;
          if (!wait_free(smem_u32(&ctrl.k_empty[s]), ((kvi / STAGES) & 1) ^ 1)) {
            ok = false;
            break;
          }
          if (!GATHER) kv_k = tile_src(begin + i, rows_k);
          load_kv(&rq.tk, rq.kg, kv_k, rows_k, sK0 + s * C::KV_BYTES, smem_u32(&ctrl.k_full[s]));
          ++k_iss;
        }
        if (i >= 1) {
          const uint32_t kvi = kv_cnt + i - 1;
          const int s = kvi % STAGES;
          if (!wait_free(smem_u32(&ctrl.v_empty[s]), ((kvi / STAGES) & 1) ^ 1)) {
            ok = false;
            break;
          }
          if (!GATHER) kv_v = tile_src(begin + i - 1, rows_v);
          load_kv(&rq.tv, rq.vg, kv_v, rows_v, sV0 + s * C::KV_BYTES, smem_u32(&ctrl.v_full[s]));
          ++v_iss;
        }
        kv_v = kv_k;
#pragma unroll
        for (int m = 0; m < BN / 32; ++m) rows_v[m] = rows_k[m];
        if constexpr (GATHER) {
          kv_k = kv_n;
#pragma unroll
          for (int m = 0; m < BN / 32; ++m) rows_k[m] = rows_n[m];
        }
      }
      kv_cnt += n;
    }
    cp_async_wait_all();
    // On an abort, let the copies already issued land before the CTA exits
    // (the last STAGES of each stream; earlier ones were consumed).
    if (*abort_flag) {
      volatile int32_t dummy = 0;
      for (uint32_t k = (k_iss > STAGES ? k_iss - STAGES : 0); k < k_iss; ++k)
        mbar_wait(smem_u32(&ctrl.k_full[k % STAGES]), (k / STAGES) & 1, &dummy, p.err);
      for (uint32_t k = (v_iss > STAGES ? v_iss - STAGES : 0); k < v_iss; ++k)
        mbar_wait(smem_u32(&ctrl.v_full[k % STAGES]), (k / STAGES) & 1, &dummy, p.err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t item_seq = 0, kv_cnt = 0, t_cnt = 0, q_cnt = 0, o_cnt = 0;
      bool ok = true;
      // Failure-path test: wait on a barrier that is never signalled, so the
      // bounded wait expires, the CTA aborts and the error word reports it.
      if (p.test_stall) ok = mbar_wait(smem_u32(&ctrl.never), 0, abort_flag, p.err, p.timeout_ns);
      while (ok) {
        const int slot = item_seq & 1;
        if (!mbar_wait(smem_u32(&ctrl.item_full[slot]), (item_seq >> 1) & 1, abort_flag, p.err, p.timeout_ns)) break;
        const int32_t it = ctrl.item_slot[slot];
        mbar_arrive(smem_u32(&ctrl.item_empty[slot]));
        ++item_seq;
        if (it < 0) break;
        const ReqParams& rq = p.req[req_of(p, it)];
        const int32_t li = it - rq.item_begin;
        const int4 i0 = __ldg(&rq.items[2 * li]);
        const int32_t n = i0.w - i0.z;
        if (n <= 0) continue;
        // tiles written by cp.async (generic proxy) are read by the tensor core
        // (async proxy): a proxy fence follows each of their full-barrier waits
        const bool gathered = GATHER || (PERM && __ldg(&rq.items[2 * li + 1]).x != 0);
        if (!mbar_wait(smem_u32(&ctrl.q_full), q_cnt & 1, abort_flag, p.err, p.timeout_ns)) break;
        ++q_cnt;
        if (gathered) fence_proxy_async_smem();
        tc_fence_after();
        if constexpr (C::Q_TMEM) {
          // Q (shared, swizzled K-major) -> TMEM, 16 columns of K per copy: lane r
          // holds row r, as the A operand of S = Q K^T expects.  The previous
          // item's QK MMAs have completed (its softmax consumed their S before
          // its last PV was issued), and the copies run ahead of this item's MMAs
          // in issue order.  The shared-memory tile is free once they land.
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tmem_cp_128x256b(tmem + C::Q_COL + kk * 8,
                             sdesc_sw128(sQ + (kk >> 2) * C::BM * 128 + (kk & 3) * 32, 16, 1024));
          mma_commit(smem_u32(&ctrl.q_empty));
        }
        // O += P V for tile j of this item
        auto issue_pv = [&](int32_t j) -> bool {
          const uint32_t t = t_cnt + j, kvi = kv_cnt + j;
          const int s = kvi % STAGES;
          const uint32_t sb = t & 1;
          if (!mbar_wait(smem_u32(&ctrl.p_full[sb]), (t >> 1) & 1, abort_flag, p.err, p.timeout_ns)) return false;
          if (!mbar_wait(smem_u32(&ctrl.v_full[s]), (kvi / STAGES) & 1, abort_flag, p.err, p.timeout_ns)) return false;
          if (gathered) fence_proxy_async_smem();
          if (j == 0) {
            if (!mbar_wait(smem_u32(&ctrl.o_empty), (o_cnt & 1) ^ 1, abort_flag, p.err, p.timeout_ns)) return false;
            ++o_cnt;
          }
          tc_fence_after();
          const uint32_t sv = sV0 + s * C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t bdesc = sdesc_sw128(sv + kk * 16 * 128, BN * 128, 1024);
            mma_bf16_ts(tmem + C::O_COL, tmem + sb * BN + kk * 8, bdesc, C::IDESC_PV,
                        (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&ctrl.v_empty[s]));
          mma_commit(smem_u32(&ctrl.pv_done));
          return true;
        };
        for (int32_t j = 0; j < n && ok; ++j) {
          const uint32_t t = t_cnt + j, kvi = kv_cnt + j;
          const int s = kvi % STAGES;
          const uint32_t sb = t & 1;
          if (!mbar_wait(smem_u32(&ctrl.k_full[s]), (kvi / STAGES) & 1, abort_flag, p.err, p.timeout_ns)) {
            ok = false;
            break;
          }
          if (gathered) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sk = sK0 + s * C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t bdesc = sdesc_sw128(sk + (kk >> 2) * BN * 128 + (kk & 3) * 32, 16, 1024);
            if constexpr (C::Q_TMEM) {
              mma_bf16_ts(tmem + sb * BN, tmem + C::Q_COL + kk * 8, bdesc, C::IDESC_QK,
                          kk > 0 ? 1u : 0u);
            } else {
              const uint64_t adesc = sdesc_sw128(sQ + (kk >> 2) * C::BM * 128 + (kk & 3) * 32, 16, 1024);
              mma_bf16_ss(tmem + sb * BN, adesc, bdesc, C::IDESC_QK, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(smem_u32(&ctrl.s_full[sb]));
          mma_commit(smem_u32(&ctrl.k_empty[s]));
          if (!C::Q_TMEM && j == n - 1) mma_commit(smem_u32(&ctrl.q_empty));
          // QK of tile j runs ahead of PV of tile j-1 (the other S buffer)
          if (j > 0 && !issue_pv(j - 1)) ok = false;
        }
        if (ok && !issue_pv(n - 1)) ok = false;
        // the item's output accumulator is complete once its last PV finishes
        if (ok) mma_commit(smem_u32(&ctrl.o_full));
        t_cnt += n;
        kv_cnt += n;
      }
      if (p.tiles_done) atomicAdd(p.tiles_done, static_cast<unsigned long long>(t_cnt));
      // every MMA issued has finished before TMEM is released
      mma_commit(smem_u32(&ctrl.final_bar));
      volatile int32_t dummy = 0;
      mbar_wait(smem_u32(&ctrl.final_bar), 0, &dummy, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- softmax warps
    const int quad = warp & 3;
    const int r = quad * 32 + lane;                    // tile row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    uint32_t item_seq = 0, t_cnt = 0, o_seq = 0, split_seq = 0;
    bool ok = true;
    while (ok) {
      const int slot = item_seq & 1;
      if (!mbar_wait(smem_u32(&ctrl.item_full[slot]), (item_seq >> 1) & 1, abort_flag, p.err, p.timeout_ns)) break;
      const int32_t it = ctrl.item_slot[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctrl.item_empty[slot]));
      ++item_seq;
      if (it < 0) break;
      const ReqParams& rq = p.req[req_of(p, it)];
      const int32_t li = it - rq.item_begin;
      const int4 i0 = __ldg(&rq.items[2 * li]);
      const int4 i1 = __ldg(&rq.items[2 * li + 1]);
      const int32_t bh = i0.x, q_tile = i0.y, begin = i0.z, n = i0.w - i0.z, layout = i1.x;
      float m_ref = -INFINITY, l = 0.f;
      // The tile entry and its boundary descriptor are fetched one tile ahead so
      // that their global-memory latency hides behind the wait for S.
      int32_t desc_next = -1, kv_next = 0;
      uint4 dn0 = make_uint4(0u, 0u, 0u, 0u), dn1 = dn0;
      if (n > 0) {
        const int2 en = __ldg(&rq.entries[begin]);
        desc_next = en.y;
        kv_next = en.x;
        if (desc_next >= 0) {
          dn0 = __ldg(&rq.descs[2 * desc_next]);
          dn1 = __ldg(&rq.descs[2 * desc_next + 1]);
        }
      }
      for (int32_t j = 0; j < n; ++j) {
        const uint32_t t = t_cnt + j;
        const uint32_t sb = t & 1;
        const int32_t desc = desc_next, kv = kv_next;
        const uint4 d0 = dn0, d1 = dn1;
        if (j + 1 < n) {
          const int2 en = __ldg(&rq.entries[begin + j + 1]);
          desc_next = en.y;
          kv_next = en.x;
          if (desc_next >= 0) {
            dn0 = __ldg(&rq.descs[2 * desc_next]);
            dn1 = __ldg(&rq.descs[2 * desc_next + 1]);
          }
        }
        if (!mbar_wait(smem_u32(&ctrl.s_full[sb]), (t >> 1) & 1, abort_flag, p.err, p.timeout_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float x[BN];
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_off + sb * BN + c0, rr);
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c0 + i] = __uint_as_float(rr[i]);
        }
        tc_wait_ld();
        // Boundary tiles: this row's column mask.  A row whose segment allows no
        // column contributes nothing (P = 0, no exponentials); a row whose
        // segment allows every in-range column needs no per-element masking.
        bool row_dead = false;
        if (GATHER && desc >= 0) {
          // list form: one BN-bit column mask per slice_m-row segment
          const bool hi = (rq.slice_m == 64) && (r >= 64);
          const uint32_t w4[4] = {hi ? d1.x : d0.x, hi ? d1.y : d0.y, hi ? d1.z : d0.z,
                                  hi ? d1.w : d0.w};
          uint32_t any = 0u, all = 0xFFFFFFFFu;
#pragma unroll
          for (int w = 0; w < BN / 32; ++w) {
            any |= w4[w];
            all &= w4[w];
          }
          if (any == 0u) {
            row_dead = true;
          } else if (all != 0xFFFFFFFFu) {
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (!((w4[c >> 5] >> (c & 31)) & 1u)) x[c] = -INFINITY;
          }
        } else if (!GATHER && desc >= 0 && (d0.x & 0xFF) == 0) {
          // band form (SVG temporal heads, temporal-major order): the row sees
          // keys whose F-token segment is within R of its own -- one interval
          const int64_t Fb = d1.w, Rb = d1.z;
          const int64_t tq = static_cast<int64_t>(q_tile) * kBM + r, seg = tq / Fb;
          const int64_t lo_a = (seg - Rb) * Fb - kv, hi_a = (seg + Rb + 1) * Fb - kv;
          const int64_t hi_n = static_cast<int64_t>(rq.N) - kv;
          const int lo = static_cast<int>(lo_a > 0 ? lo_a : 0);
          const int hi = static_cast<int>(hi_a < BN ? (hi_a < hi_n ? hi_a : hi_n) : (BN < hi_n ? BN : hi_n));
          if (tq >= rq.N || lo >= hi) {
            row_dead = true;
          } else if (lo > 0 || hi < BN) {
            uint32_t words[BN / 32];
#pragma unroll
            for (int w = 0; w < BN / 32; ++w) words[w] = 0u;
            add_range<BN>(words, lo, hi);
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (!((words[c >> 5] >> (c & 31)) & 1u)) x[c] = -INFINITY;
          }
        } else if (desc >= 0) {
          const int n_r = d0.x & 0xFF, n_c = (d0.x >> 8) & 0xFF;
          int rs = 0;
#pragma unroll
          for (int k = 1; k < 8; ++k)
            if (k < n_r && static_cast<int>(desc_byte(d0, d1, 2 + k)) <= r) rs = k;
          const uint64_t bits = (static_cast<uint64_t>(d1.w) << 32) | d1.z;
          const uint32_t all_c = (1u << n_c) - 1u;
          const uint32_t rb = static_cast<uint32_t>(bits >> (rs * 8)) & all_c;
          const int c_end = static_cast<int>(desc_byte(d0, d1, 10 + n_c));
          if (rb == 0u) {
            row_dead = true;
          } else if (rb != all_c || c_end < BN) {
            uint32_t words[BN / 32];
#pragma unroll
            for (int w = 0; w < BN / 32; ++w) words[w] = 0u;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              if (c < n_c && ((rb >> c) & 1u))
                add_range<BN>(words, static_cast<int>(desc_byte(d0, d1, 10 + c)),
                              static_cast<int>(desc_byte(d0, d1, 11 + c)));
            }
#pragma unroll
            for (int c = 0; c < BN; ++c)
              if (!((words[c >> 5] >> (c & 31)) & 1u)) x[c] = -INFINITY;
          }
        }
        // P = 2^(x * scale - m_use) for the row, written to TMEM as bf16 pairs;
        // returns the row sum.  With track_max the same pass also takes the
        // row maximum of x (three-input max over column pairs).
        auto p_pass = [&](float m_use, bool track_max, float& mx) -> float {
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f, s5 = 0.f, s6 = 0.f, s7 = 0.f;
#pragma unroll
          for (int c0 = 0; c0 < BN; c0 += 64) {
            uint32_t pk[32];
            if (row_dead) {
#pragma unroll
              for (int i = 0; i < 32; ++i) pk[i] = 0u;
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float x0 = x[c0 + 2 * i], x1 = x[c0 + 2 * i + 1];
                float y0, y1;
                fma2(y0, y1, x0, x1, p.scale_log2, -m_use);
                const float a = ex2_approx(y0), b = ex2_approx(y1);
                if ((i & 3) == 0) add2(s0, s1, a, b);
                else if ((i & 3) == 1) add2(s2, s3, a, b);
                else if ((i & 3) == 2) add2(s4, s5, a, b);
                else add2(s6, s7, a, b);
                if (track_max) mx = max3f(mx, x0, x1);
                pk[i] = pack_bf16x2(a, b);
              }
            }
            tmem_st32(tmem + lane_off + sb * BN + c0 / 2, pk);
          }
          return ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
        };
        // A row with no finite maximum yet takes its reference maximum from this
        // tile first.  Otherwise P is computed against the current reference
        // maximum while the tile maximum is taken in the same pass; only if the
        // maximum grew by more than the threshold is P recomputed (whole warp,
        // since the TMEM store is warp-collective) and O rescaled.
        const bool first = (m_ref == -INFINITY);
        if (first && !row_dead) {
          float a0 = fmaxf(x[0], x[1]), a1 = fmaxf(x[2], x[3]), a2 = fmaxf(x[4], x[5]),
                a3 = fmaxf(x[6], x[7]);
#pragma unroll
          for (int c = 8; c < BN; c += 8) {
            a0 = max3f(a0, x[c], x[c + 1]);
            a1 = max3f(a1, x[c + 2], x[c + 3]);
            a2 = max3f(a2, x[c + 4], x[c + 5]);
            a3 = max3f(a3, x[c + 6], x[c + 7]);
          }
          m_ref = fmaxf(max3f(a0, a1, a2), a3) * p.scale_log2;   // stays -inf if all masked
        }
        float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        float mx = -INFINITY;
        float rowsum = p_pass(m_use, true, mx);
        bool fix = false;
        float alpha = 1.f;
        if (!first && !row_dead) {
          const float mt = mx * p.scale_log2;
          if (mt > m_ref + kRescaleThreshold) {
            fix = true;
            alpha = ex2_approx(m_ref - mt);
            m_ref = mt;
            m_use = mt;
          }
        }
        if (__any_sync(0xFFFFFFFFu, fix)) {
          float unused = 0.f;
          rowsum = p_pass(m_use, false, unused);
        }
        l = l * alpha + rowsum;
        // Rescale O (the sum over earlier tiles) when the reference maximum grew.
        // Rows that had no finite maximum before hold O = 0 and need nothing.
        const bool fix_o = fix && j > 0;
        if (__any_sync(0xFFFFFFFFu, fix_o)) {
          if (!mbar_wait(smem_u32(&ctrl.pv_done), (t - 1) & 1, abort_flag, p.err, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float f = fix_o ? alpha : 1.f;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t rr[32];
            tmem_ld32(tmem + lane_off + C::O_COL + c0, rr);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * f);
            tmem_st32(tmem + lane_off + C::O_COL + c0, rr);
          }
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl.p_full[sb]));
      }
      if (!ok) break;
      t_cnt += n;
      // ----------------------------------------------------------- epilogue
      const int32_t gr = q_tile * kBM + r;
      const bool valid = gr < rq.N;
      const int32_t orow = (PERM && layout) ? unpermute(gr, rq.F, rq.S) : gr;
      const size_t obase = (static_cast<size_t>(bh) * rq.N + (valid ? orow : 0)) * D;
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      if (i1.z > 1) {
        // split-KV unit (part i1.w of the i1.z parts of work item i1.y): its
        // normalised partial row O / l (fp32) and lse (base 2) go to the
        // plan's workspace; the last part of the item to finish merges them
        const int64_t unit = static_cast<int64_t>(i1.y) * i1.z + i1.w;
        // layout [unit][d / 4][row] of float4: a warp's rows are adjacent
        float4* po = reinterpret_cast<float4*>(rq.part_o + unit * kBM * D) + r;
        if (n > 0) {
          if (!mbar_wait(smem_u32(&ctrl.o_full), o_seq & 1, abort_flag, p.err, p.timeout_ns)) break;
          ++o_seq;
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t rr[32];
            tmem_ld32(tmem + lane_off + C::O_COL + c0, rr);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              po[(c0 / 4 + i) * kBM] =
                  make_float4(__uint_as_float(rr[4 * i]) * inv_l, __uint_as_float(rr[4 * i + 1]) * inv_l,
                              __uint_as_float(rr[4 * i + 2]) * inv_l, __uint_as_float(rr[4 * i + 3]) * inv_l);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctrl.o_empty));
        } else {
#pragma unroll
          for (int i = 0; i < D / 4; ++i) po[i * kBM] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        rq.part_lse[unit * kBM + r] = (l > 0.f) ? m_ref + __log2f(l) : -INFINITY;
        __threadfence();
        // every row of the part is written: count the part
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl.split_bar));
        if (!mbar_wait(smem_u32(&ctrl.split_bar), split_seq & 1, abort_flag, p.err, p.timeout_ns)) break;
        ++split_seq;
        if (r == 0) ctrl.split_last = (atomicAdd(rq.part_cnt + i1.y, 1) == i1.z - 1) ? 1 : 0;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl.split_bar));
        if (!mbar_wait(smem_u32(&ctrl.split_bar), split_seq & 1, abort_flag, p.err, p.timeout_ns)) break;
        ++split_seq;
        if (ctrl.split_last && valid) {
          __threadfence();
          const int64_t u0 = static_cast<int64_t>(i1.y) * i1.z;
          float w[4], M = -INFINITY;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            w[q] = (q < i1.z) ? __ldcg(rq.part_lse + (u0 + q) * kBM + r) : -INFINITY;
            M = fmaxf(M, w[q]);
          }
          float L = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            w[q] = (M == -INFINITY) ? 0.f : ex2_approx(w[q] - M);   // ex2(-inf) = 0
            L += w[q];
          }
          const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) w[q] *= inv;
          // every part's two float4 of a chunk are loaded together (parts past
          // i1.z load nothing and weigh 0), two chunks in flight
          const float4* src[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            src[q] = reinterpret_cast<const float4*>(rq.part_o + (u0 + (q < i1.z ? q : 0)) * kBM * D) + r;
          uint4* dst = reinterpret_cast<uint4*>(rq.out + obase);
#pragma unroll 2
          for (int c = 0; c < D / 8; ++c) {
            float4 x[4][2];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const bool on = q < i1.z;
              x[q][0] = on ? __ldcg(src[q] + (2 * c) * kBM) : make_float4(0.f, 0.f, 0.f, 0.f);
              x[q][1] = on ? __ldcg(src[q] + (2 * c + 1) * kBM) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[0] += w[q] * x[q][0].x; acc[1] += w[q] * x[q][0].y;
              acc[2] += w[q] * x[q][0].z; acc[3] += w[q] * x[q][0].w;
              acc[4] += w[q] * x[q][1].x; acc[5] += w[q] * x[q][1].y;
              acc[6] += w[q] * x[q][1].z; acc[7] += w[q] * x[q][1].w;
            }
            dst[c] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
          }
          rq.lse[static_cast<size_t>(bh) * rq.N + orow] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
        }
        continue;
      }
      if (n > 0) {
        // o_full completes once per non-empty item, after its last PV; the next
        // item's first PV waits for o_empty, so the phases cannot run ahead.
        if (!mbar_wait(smem_u32(&ctrl.o_full), o_seq & 1, abort_flag, p.err, p.timeout_ns)) break;
        ++o_seq;
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_off + C::O_COL + c0, rr);
          tc_wait_ld();
          if (valid) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * inv_l,
                                  __uint_as_float(rr[2 * i + 1]) * inv_l);
            uint4* dst = reinterpret_cast<uint4*>(rq.out + obase + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl.o_empty));
      } else if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(rq.out + obase);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (valid)
        rq.lse[static_cast<size_t>(bh) * rq.N + orow] =
            (l > 0.f) ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int BN, int STAGES, int CTAS, int MODE, int MAXR>
tsr_status launch_variant(const FwdParamsT<MAXR>& prm, int n_items, int device, cudaStream_t stream) {
  using C = Cfg<D, BN, STAGES, CTAS>;
  auto kern = bsa_fwd_kernel<D, BN, STAGES, CTAS, MODE, MAXR>;
  static bool attr_set[64] = {false};
  if (device < 0 || device >= 64 || !attr_set[device]) {
    TSR_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM));
    if (device >= 0 && device < 64) attr_set[device] = true;
  }
  const int grid = std::min(n_items, num_sms(device) * CTAS);
  if (grid <= 0) return TSR_OK;
  kern<<<grid, 192, C::SMEM, stream>>>(prm);
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

// Kernel variants compiled into the library: (d, BN, stages, CTAs per SM).  The
// contiguous list is compiled for kModeTma and kModePerm, the gathered one for
// kModeList.
#define TSR_VARIANTS_CONTIGUOUS(X) \
  X(128, 128, 3, 1) X(128, 128, 2, 1) X(128, 64, 4, 1) X(128, 64, 2, 2) \
  X(64, 128, 4, 1) X(64, 64, 4, 1) X(64, 64, 3, 2)
#define TSR_VARIANTS_GATHERED(X) X(128, 128, 3, 1) X(128, 64, 2, 2) X(64, 128, 4, 1) X(64, 64, 3, 2)
// Variants also compiled for batched launches (the table's choices at long
// sequences), in every mode.
#define TSR_VARIANTS_BATCH(X) X(128, 64, 2, 2) X(64, 64, 3, 2)

constexpr int vkey(int d, int bn, int stages, int ctas) {
  return d * 100000 + bn * 100 + stages * 10 + ctas;
}

// Launch the compiled variant `key` of one mode (each defined in its own
// translation unit so the modes compile in parallel); TSR_ERR_UNSUPPORTED when
// that mode has no such variant.
tsr_status launch_mode_tma(const FwdParams& prm, int key, int n_items, int device, cudaStream_t stream);
tsr_status launch_mode_perm(const FwdParams& prm, int key, int n_items, int device, cudaStream_t stream);
tsr_status launch_mode_list(const FwdParams& prm, int key, int n_items, int device, cudaStream_t stream);
tsr_status launch_mode_tma(const FwdParamsBatch& prm, int key, int n_items, int device,
                           cudaStream_t stream);
tsr_status launch_mode_perm(const FwdParamsBatch& prm, int key, int n_items, int device,
                            cudaStream_t stream);
tsr_status launch_mode_list(const FwdParamsBatch& prm, int key, int n_items, int device,
                            cudaStream_t stream);

}  // namespace fwd
}  // namespace tsr
