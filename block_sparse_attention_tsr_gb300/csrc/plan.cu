// plan.cu -- physical mapping and task organisation on the GPU.
//
// Tessera abstract: a mapping layer keeps, merges or cuts logical blocks into
// physical tiles that suit the mask and the GPU, and a task layer groups the
// tiles into GPU tasks.  Here a physical tile is bm query rows by BN keys: 128
// rows (the tcgen05 M = 128 datapath with queries on M) by 64 or 128 keys, or,
// for key-major plans, 64 rows by 64 keys (two such tiles of a query block are
// computed together with 128 keys on M):
//   * logical blocks of the tile's size map one-to-one (kept),
//   * smaller blocks (32, 64, frames of 21 tokens) are merged into a tile,
//   * larger blocks (256, 1,560-token frames) are cut into several tiles.
// Each tile is classified from the logical segments that overlap it:
//   empty    -> dropped (never loaded or computed),
//   full     -> every element allowed and every key in range: no masking,
//   boundary -> mixed, or crossing N: a 32-byte descriptor (row segments x
//               column segments bit grid) drives element masking.
// (Splash digest, "Splash Attention": skip empty tiles, exact masking only on
// boundary tiles.)  The task layer gives every bm-row query tile one work item
// holding its tiles in key order; items are ordered longest first so that a
// persistent grid finishes evenly, and the regime table picks the orientation,
// tile width and pipeline depth.  Three kernels: count (both tile widths at one
// height, so either width's totals are at hand once the regime is known), schedule
// (one block: prefix sums + longest-first order), emit (tiles and
// descriptors); then the attention launch list (without SVG temporal heads that
// run by spatial position) and the split-KV units.
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace tsr {

namespace {

constexpr int kMaxSeg = 8;

// Logical segments of one axis (0 = queries, 1 = keys) that overlap tokens
// [t0, t1) of head h.  ids[] receive segment ids, starts[] the first token of
// each relative to t0; entries from the count on hold t1 - t0 (so starts[n] =
// t1 - t0).  Returns the count, or -1 if more than kMaxSeg segments overlap.
// The overlapping segments are consecutive ids, so every array index below is
// a compile-time constant and the arrays stay in registers.
__device__ __forceinline__ int tile_segments(const MaskDev& m, int h, int axis, int t0, int t1,
                                             int (&ids)[kMaxSeg], int (&starts)[kMaxSeg + 1]) {
  int n = 0;
  bool more = false;                 // a (kMaxSeg + 1)-th segment overlaps
  if (m.kind == TSR_MASK_SEGMENTS) {
    const int32_t* bd = axis ? m.k_bounds : m.q_bounds;
    const int ns = axis ? m.n_kseg : m.n_qseg;
    int lo = 0, hi = ns - 1;  // last segment whose start <= t0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (bd[mid] <= t0) lo = mid; else hi = mid - 1;
    }
#pragma unroll
    for (int k = 0; k < kMaxSeg; ++k) {
      const int id = lo + k;
      const int b = id < ns ? bd[id] : t1;
      const bool v = b < t1;
      ids[k] = id;
      starts[k] = v ? max(b, t0) - t0 : t1 - t0;
      n += v;
    }
    more = lo + kMaxSeg < ns && bd[lo + kMaxSeg] < t1;
  } else {
    int size;
    if (m.kind == TSR_MASK_UNIFORM) size = axis ? m.bk : m.bq;
    else size = (m.head_kind[h] == TSR_HEAD_TEMPORAL) ? m.F : m.S;  // SVG
    const int first = t0 / size;
#pragma unroll
    for (int k = 0; k < kMaxSeg; ++k) {
      const int id = first + k;
      const bool v = id * size < t1;
      ids[k] = id;
      starts[k] = v ? max(id * size, t0) - t0 : t1 - t0;
      n += v;
    }
    more = (first + kMaxSeg) * size < t1;
  }
  starts[kMaxSeg] = t1 - t0;
  return more ? -1 : n;
}

__device__ __forceinline__ bool seg_allowed(const MaskDev& m, int bh, int h, int qid, int kid,
                                            int64_t nqs, int64_t nks) {
  if (m.kind == TSR_MASK_SVG) {
    if (m.head_kind[h] == TSR_HEAD_TEMPORAL) return abs(qid - kid) <= m.R;  // index within R
    return qid == kid || kid == 0;                                // same frame, or frame 0
  }
  return m.blocks[(static_cast<int64_t>(bh) * nqs + qid) * nks + kid] != 0;
}

struct RowSegs {
  int n;
  int ids[kMaxSeg];
  int starts[kMaxSeg + 1];
  int q0, q1;                // the tile's query rows [q0, q1)
};

// SVG temporal heads in temporal-major order: row t' may see keys whose
// F-token segment is within R of its own, |t'/F - j/F| <= R.  Each row's keys
// form one interval and the rows' intervals grow with the row, so a tile is
// empty, full or "band" from its first and last rows.  Band tiles get a
// descriptor with n_r = 0 and bits = F << 32 | R; the kernel masks each row to
// its interval (any frame count: no per-tile segment limit).
__device__ int classify_band(const MaskDev& m, int q0, int q1, int k0, int bn, tsr_tile_desc* desc) {
  if (k0 >= m.N) return 0;
  const int64_t F = m.F, R = m.R, k1 = min(m.N, k0 + bn);
  const int64_t s_first = q0 / F, s_last = (q1 - 1) / F;
  const int64_t lo_a = (s_first - R) * F, hi_a = (s_last + R + 1) * F;
  const int64_t lo_u = lo_a > 0 ? lo_a : 0, hi_u = hi_a < m.N ? hi_a : m.N;
  if (k1 <= lo_u || k0 >= hi_u) return 0;
  if (k0 + bn <= m.N && (s_first + R + 1) * F >= k0 + bn && (s_last - R) * F <= k0) return 1;
  if (desc) {
    memset(desc, 0, sizeof(*desc));
    desc->bits = (static_cast<uint64_t>(m.F) << 32) | static_cast<uint32_t>(m.R);
  }
  return 2;
}

// 0 empty, 1 full, 2 boundary, -1 unsupported.  desc is filled for boundary tiles.
__device__ int classify(const MaskDev& m, int bh, int h, const RowSegs& rs, int k0, int bn,
                        int64_t nqs, int64_t nks, tsr_tile_desc* desc) {
  if (m.kind == TSR_MASK_SVG && m.head_kind[h] == TSR_HEAD_TEMPORAL)
    return classify_band(m, rs.q0, rs.q1, k0, bn, desc);
  if (k0 >= m.N) return 0;
  const int k1 = min(m.N, k0 + bn);
  int cid[kMaxSeg], cst[kMaxSeg + 1];
  const int nc = tile_segments(m, h, 1, k0, k1, cid, cst);
  if (nc < 0 || rs.n < 0) return -1;
  uint64_t bits = 0;
  bool any = false, all = true;
#pragma unroll
  for (int r = 0; r < kMaxSeg; ++r) {
    if (r >= rs.n) break;
#pragma unroll
    for (int c = 0; c < kMaxSeg; ++c) {
      if (c >= nc) break;
      const bool a = seg_allowed(m, bh, h, rs.ids[r], cid[c], nqs, nks);
      any |= a;
      all &= a;
      if (a) bits |= 1ull << (r * 8 + c);
    }
  }
  if (!any) return 0;
  if (all && k1 - k0 == bn) return 1;
  if (desc) {
    // the 32-byte descriptor as 8 words: n_r, n_c, r_start[8], c_start[9], pad,
    // bits (byte offsets 0, 1, 2..9, 10..18, 19..23, 24..31)
    uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    auto put = [&](int byte, uint32_t v) { w[byte >> 2] |= (v & 0xFFu) << ((byte & 3) * 8); };
    put(0, static_cast<uint32_t>(rs.n));
    put(1, static_cast<uint32_t>(nc));
#pragma unroll
    for (int r = 0; r < kMaxSeg; ++r)
      if (r < rs.n) put(2 + r, static_cast<uint32_t>(rs.starts[r]));
#pragma unroll
    for (int c = 0; c <= kMaxSeg; ++c)
      if (c <= nc) put(10 + c, static_cast<uint32_t>(cst[c]));
    w[6] = static_cast<uint32_t>(bits);
    w[7] = static_cast<uint32_t>(bits >> 32);
    static_assert(sizeof(tsr_tile_desc) == 32, "descriptor size");
    memcpy(desc, w, 32);
  }
  return 2;
}

// Key tiles of width w that can hold an allowed key for query rows [q0, q1),
// as up to two ascending, disjoint tile-index ranges [t0, t1).  SVG spatial
// heads: frame 0 and the rows' own frames; SVG temporal heads (temporal-major
// order): the F-token segments within the radius of the rows' own.  Every
// other tile is empty for these rows, so count and emit skip it.  Other mask
// kinds: all tiles.
struct KeyWindow {
  int n;
  int t0[2], t1[2];
  __device__ int size() const { return (t1[0] - t0[0]) + (n > 1 ? t1[1] - t0[1] : 0); }
  __device__ int tile(int i) const { return i < t1[0] - t0[0] ? t0[0] + i : t0[1] + i - (t1[0] - t0[0]); }
};

__device__ KeyWindow key_window(const MaskDev& m, int h, int q0, int q1, int w) {
  int lo0 = 0, hi0 = m.N, lo1 = 0, hi1 = 0;   // token ranges
  if (m.kind == TSR_MASK_SVG) {
    if (m.head_kind[h] == TSR_HEAD_TEMPORAL) {
      const int64_t s0 = q0 / m.F - m.R, s1 = (q1 - 1) / m.F + 1 + static_cast<int64_t>(m.R);
      lo0 = static_cast<int>((s0 > 0 ? s0 : 0) * m.F);
      hi0 = static_cast<int>(s1 * m.F < m.N ? s1 * m.F : m.N);
    } else {
      hi0 = m.S;
      lo1 = (q0 / m.S) * m.S;
      hi1 = min(m.N, ((q1 - 1) / m.S + 1) * m.S);
    }
  }
  KeyWindow kw;
  kw.n = 1;
  kw.t0[0] = lo0 / w;
  kw.t1[0] = (hi0 + w - 1) / w;
  kw.t0[1] = kw.t1[1] = 0;
  if (hi1 > lo1) {
    const int b0 = lo1 / w, b1 = (hi1 + w - 1) / w;
    if (b0 <= kw.t1[0]) {
      kw.t1[0] = max(kw.t1[0], b1);
    } else {
      kw.n = 2;
      kw.t0[1] = b0;
      kw.t1[1] = b1;
    }
  }
  return kw;
}

__device__ void grid_dims(const MaskDev& m, int64_t* nqs, int64_t* nks) {
  if (m.kind == TSR_MASK_UNIFORM) {
    *nqs = (m.N + m.bq - 1) / m.bq;
    *nks = (m.N + m.bk - 1) / m.bk;
  } else if (m.kind == TSR_MASK_SEGMENTS) {
    *nqs = m.n_qseg;
    *nks = m.n_kseg;
  } else {
    *nqs = *nks = 0;
  }
}

// UNIFORM masks whose query tiles lie inside one logical row block (bq a
// multiple of the tile height) and whose 64-key sub-tiles lie inside one
// logical column block (bk a multiple of 64): a sub-tile is allowed iff its one
// logical block is, and full iff also inside [0, N).  The count and emit
// kernels then read the row of logical blocks directly instead of classifying
// segment grids (same results as classify(); the ragged last key tile still
// goes through classify() for its descriptor).
__device__ __forceinline__ bool aligned_uniform(const MaskDev& m, int bm, int bn) {
  return m.kind == TSR_MASK_UNIFORM && m.bq % bm == 0 && m.bk % bn == 0;
}

// Per query tile: [0] tiles at BN=64, [1] boundary tiles at BN=64, [2] tiles at
// BN=128, [3] boundary at BN=128.  Totals: the same four sums, then [4], [5] the
// longest item at BN=64 / 128, [6] allowed logical blocks.
__global__ void plan_count_kernel(MaskDev m, int32_t nqt, int32_t bm, int32_t* cnt,
                                  unsigned long long* tot, uint32_t* err) {
  __shared__ unsigned long long bsum[6];
  if (threadIdx.x < 6) bsum[threadIdx.x] = 0;
  __syncthreads();
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n_items = static_cast<int64_t>(m.B) * m.H * nqt;
  if (warp < n_items) {
    const int bh = static_cast<int>(warp / nqt), qt = static_cast<int>(warp % nqt), h = bh % m.H;
    RowSegs rs;
    rs.q0 = qt * bm;
    rs.q1 = min(m.N, qt * bm + bm);
    rs.n = (m.kind == TSR_MASK_SVG && m.head_kind[h] == TSR_HEAD_TEMPORAL)
               ? 0
               : tile_segments(m, h, 0, rs.q0, rs.q1, rs.ids, rs.starts);
    int64_t nqs, nks;
    grid_dims(m, &nqs, &nks);
    const KeyWindow kw = key_window(m, h, rs.q0, rs.q1, 128);
    const int n_kt = kw.size();
    int e64 = 0, b64 = 0, e128 = 0, b128 = 0;
    bool bad = false;
    if (aligned_uniform(m, bm, 64)) {
      // 64-key sub-tiles s < ceil(N / 64), 16 consecutive ones per lane (their
      // loads issued together); 128-key tile i = sub-tiles 2i and 2i + 1
      const uint8_t* row = m.blocks + (static_cast<int64_t>(bh) * nqs + rs.q0 / m.bq) * nks;
      const int n64 = (m.N + 63) >> 6, per = m.bk >> 6;
      for (int base = 0; base < n64; base += 32 * 16) {
        const int s0 = base + lane * 16;
        uint32_t on = 0, full = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int sj = s0 + j;
          if (sj < n64 && __ldg(row + sj / per) != 0) {
            on |= 1u << j;
            if ((sj + 1) * 64 <= m.N) full |= 1u << j;
          }
        }
        const uint32_t pair_on = (on | (on >> 1)) & 0x5555u, pair_full = (full & (full >> 1)) & 0x5555u;
        e64 += __popc(on);
        b64 += __popc(on & ~full);
        e128 += __popc(pair_on);
        b128 += __popc(pair_on & ~pair_full);
      }
    } else
    for (int i = lane; i < n_kt; i += 32) {
      const int kt = kw.tile(i);
      const int ca = classify(m, bh, h, rs, kt * 128, 64, nqs, nks, nullptr);
      const int cb = classify(m, bh, h, rs, kt * 128 + 64, 64, nqs, nks, nullptr);
      if (ca < 0 || cb < 0) {
        bad = true;
        continue;
      }
      e64 += (ca != 0) + (cb != 0);
      b64 += (ca == 2) + (cb == 2);
      if (ca != 0 || cb != 0) {
        ++e128;
        if (!(ca == 1 && cb == 1)) ++b128;
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      e64 += __shfl_xor_sync(0xFFFFFFFFu, e64, o);
      b64 += __shfl_xor_sync(0xFFFFFFFFu, b64, o);
      e128 += __shfl_xor_sync(0xFFFFFFFFu, e128, o);
      b128 += __shfl_xor_sync(0xFFFFFFFFu, b128, o);
    }
    if (__any_sync(0xFFFFFFFFu, bad)) {
      if (lane == 0) atomicOr(err, DEV_ERR_UNSUPPORTED);
    } else if (lane == 0) {
      cnt[0 * n_items + warp] = e64;
      cnt[1 * n_items + warp] = b64;
      cnt[2 * n_items + warp] = e128;
      cnt[3 * n_items + warp] = b128;
      atomicAdd(&bsum[0], static_cast<unsigned long long>(e64));
      atomicAdd(&bsum[1], static_cast<unsigned long long>(b64));
      atomicAdd(&bsum[2], static_cast<unsigned long long>(e128));
      atomicAdd(&bsum[3], static_cast<unsigned long long>(b128));
      atomicMax(&bsum[4], static_cast<unsigned long long>(e64));
      atomicMax(&bsum[5], static_cast<unsigned long long>(e128));
    }
  }
  // one set of global atomics per block
  __syncthreads();
  if (threadIdx.x < 4) {
    if (bsum[threadIdx.x]) atomicAdd(&tot[threadIdx.x], bsum[threadIdx.x]);
  } else if (threadIdx.x < 6) {
    atomicMax(&tot[threadIdx.x], bsum[threadIdx.x]);
  }
}

// Number of allowed logical blocks (density for the regime table): 16 bytes
// per load where the array is 16-byte aligned, single bytes for the rest.
__global__ void logical_count_kernel(const uint8_t* blocks, int64_t n, unsigned long long* out) {
  unsigned long long c = 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t head = min(n, static_cast<int64_t>((16 - (reinterpret_cast<uintptr_t>(blocks) & 15)) & 15));
  const int64_t n16 = (n - head) >> 4;
  const uint4* v = reinterpret_cast<const uint4*>(blocks + head);
  auto nz = [](uint32_t w) {   // non-zero bytes of a word
    return __popc(((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu | w) & 0x80808080u);
  };
  for (int64_t i = t; i < n16; i += stride) {
    const uint4 x = __ldg(v + i);
    c += nz(x.x) + nz(x.y) + nz(x.z) + nz(x.w);
  }
  for (int64_t i = t; i < head; i += stride) c += blocks[i] != 0;
  for (int64_t i = head + 16 * n16 + t; i < n; i += stride) c += blocks[i] != 0;
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
  if ((threadIdx.x & 31) == 0 && c) atomicAdd(out, c);
}

// Exclusive scans of a[0, n) and, if b is not null, b[0, n) with one block
// (a multiple of 32 threads, at most 1024): each thread sums a contiguous run
// of ceil(n / T) values, warp shuffles and one shared array of warp totals give
// every run its offset, and the run is written back (out may equal in).
__device__ void block_scan_runs(const int32_t* a, const int32_t* b, int32_t* oa, int32_t* ob,
                                int64_t n, int32_t* wa, int32_t* wb) {
  const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = T >> 5;
  const int64_t per = (n + T - 1) / T;
  const int64_t lo = min(n, static_cast<int64_t>(tid) * per), hi = min(n, lo + per);
  constexpr int kBatch = 8;                    // loads issued together (latency-bound block)
  int32_t sa = 0, sb = 0;
  for (int64_t i0 = lo; i0 < hi; i0 += kBatch) {
    int32_t va[kBatch], vb[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      va[j] = i0 + j < hi ? a[i0 + j] : 0;
      vb[j] = (b && i0 + j < hi) ? b[i0 + j] : 0;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      sa += va[j];
      sb += vb[j];
    }
  }
  int32_t xa = sa, xb = sb;                    // inclusive scan over the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t ya = __shfl_up_sync(0xFFFFFFFFu, xa, o), yb = __shfl_up_sync(0xFFFFFFFFu, xb, o);
    if (lane >= o) {
      xa += ya;
      xb += yb;
    }
  }
  if (lane == 31) {
    wa[warp] = xa;
    wb[warp] = xb;
  }
  __syncthreads();
  if (warp == 0) {                             // exclusive scan of the warp totals
    const int32_t va = lane < nw ? wa[lane] : 0, vb = lane < nw ? wb[lane] : 0;
    int32_t ia = va, ib = vb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t ya = __shfl_up_sync(0xFFFFFFFFu, ia, o), yb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
      if (lane >= o) {
        ia += ya;
        ib += yb;
      }
    }
    if (lane < nw) {
      wa[lane] = ia - va;
      wb[lane] = ib - vb;
    }
  }
  __syncthreads();
  int32_t ra = wa[warp] + xa - sa, rb = wb[warp] + xb - sb;
  for (int64_t i0 = lo; i0 < hi; i0 += kBatch) {
    int32_t va[kBatch], vb[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      va[j] = i0 + j < hi ? a[i0 + j] : 0;
      vb[j] = (b && i0 + j < hi) ? b[i0 + j] : 0;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (i0 + j < hi) {
        oa[i0 + j] = ra;
        if (b) ob[i0 + j] = rb;
      }
      ra += va[j];
      rb += vb[j];
    }
  }
  __syncthreads();
}

// Largest LPT histogram kept in shared memory (32-bit buckets).
constexpr int64_t kSharedBuckets = 12288;

// One block: tile offsets, descriptor offsets and the work items.  With lpt the
// items are ordered by head group (group_heads consecutive (b, h) per group,
// sized so a group's K and V stay in L2), and longest first inside a group
// (counting sort over n_groups x (max_len + 1) buckets, in shared memory when
// there are at most kSharedBuckets, else in `hist`).
__global__ void __launch_bounds__(1024) plan_schedule_kernel(
    const int32_t* cnt_e, const int32_t* cnt_b, int64_t n_items, int32_t nqt, int32_t H,
    const int8_t* head_kind, int32_t is_svg, int32_t max_len, int32_t lpt, int32_t group_heads,
    int64_t n_buckets, int32_t* ebegin, int32_t* dbegin, int32_t* hist, int4* items) {
  extern __shared__ int32_t shist[];
  __shared__ int32_t wa[32], wb[32];
  block_scan_runs(cnt_e, cnt_b, ebegin, dbegin, n_items, wa, wb);
  // item indices fit 32 bits (the planner refuses more than 2^30 items), so
  // the divisions below are 32-bit
  const int T = blockDim.x, tid = threadIdx.x;
  const uint32_t per_group = static_cast<uint32_t>(group_heads) * static_cast<uint32_t>(nqt);
  const uint32_t unqt = static_cast<uint32_t>(nqt), n32 = static_cast<uint32_t>(n_items);
  int32_t* hb = (n_buckets <= kSharedBuckets) ? shist : hist;
  constexpr int kBatch = 4;                    // items whose loads are issued together
  if (lpt) {
    for (int64_t i = tid; i < n_buckets; i += T) hb[i] = 0;
    __syncthreads();
    for (uint32_t i0 = tid; i0 < n32; i0 += kBatch * T) {
      int32_t len[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) len[j] = i0 + j * T < n32 ? cnt_e[i0 + j * T] : 0;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const uint32_t i = i0 + j * T;
        if (i < n32) atomicAdd(&hb[(i / per_group) * (max_len + 1) + (max_len - len[j])], 1);
      }
    }
    __syncthreads();
    block_scan_runs(hb, nullptr, hb, nullptr, n_buckets, wa, wb);   // bucket start positions
  }
  for (uint32_t i0 = tid; i0 < n32; i0 += kBatch * T) {
    int32_t len[kBatch], beg[kBatch];
    int8_t kind[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const uint32_t i = i0 + j * T;
      const bool ok = i < n32;
      len[j] = ok ? cnt_e[i] : 0;
      beg[j] = ok ? ebegin[i] : 0;
      kind[j] = (ok && is_svg) ? head_kind[(i / unqt) % static_cast<uint32_t>(H)] : 0;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const uint32_t i = i0 + j * T;
      if (i >= n32) break;
      const int64_t pos =
          lpt ? atomicAdd(&hb[(i / per_group) * (max_len + 1) + (max_len - len[j])], 1) : i;
      const int32_t bh = static_cast<int32_t>(i / unqt), qt = static_cast<int32_t>(i % unqt);
      const int32_t layout = kind[j] == TSR_HEAD_TEMPORAL ? 1 : 0;
      items[2 * pos] = make_int4(bh, qt, beg[j], beg[j] + len[j]);
      items[2 * pos + 1] = make_int4(layout, 0, 0, 0);
    }
  }
}

// Dynamic shared memory of a plan_schedule_kernel launch.
size_t schedule_smem(int64_t n_buckets) {
  return n_buckets <= kSharedBuckets ? static_cast<size_t>(n_buckets) * 4 : 0;
}

__global__ void plan_emit_kernel(MaskDev m, int32_t nqt, int32_t bm, int32_t bn,
                                 const int32_t* ebegin, const int32_t* dbegin, int2* entries,
                                 tsr_tile_desc* descs) {
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n_items = static_cast<int64_t>(m.B) * m.H * nqt;
  if (warp >= n_items) return;
  const int bh = static_cast<int>(warp / nqt), qt = static_cast<int>(warp % nqt), h = bh % m.H;
  RowSegs rs;
  rs.q0 = qt * bm;
  rs.q1 = min(m.N, qt * bm + bm);
  rs.n = (m.kind == TSR_MASK_SVG && m.head_kind[h] == TSR_HEAD_TEMPORAL)
             ? 0
             : tile_segments(m, h, 0, rs.q0, rs.q1, rs.ids, rs.starts);
  int64_t nqs, nks;
  grid_dims(m, &nqs, &nks);
  const KeyWindow kw = key_window(m, h, rs.q0, rs.q1, bn);
  const int n_kt = kw.size();
  int32_t e_pos = ebegin[warp], d_pos = dbegin[warp];
  if (aligned_uniform(m, bm, bn)) {
    // tiles kt < n_kt, 16 consecutive ones per lane (their loads issued
    // together); an allowed tile is full inside [0, N), else it is the ragged
    // last tile, the item's one boundary tile (classify() builds its descriptor)
    const uint8_t* row = m.blocks + (static_cast<int64_t>(bh) * nqs + rs.q0 / m.bq) * nks;
    const int per = m.bk / bn;
    for (int base = 0; base < n_kt; base += 32 * 16) {
      const int t0 = base + lane * 16;
      uint32_t on = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (t0 + j < n_kt && __ldg(row + (t0 + j) / per) != 0) on |= 1u << j;
      const int cnt = __popc(on);
      int x = cnt;                                       // inclusive scan over the lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      int32_t at = e_pos + x - cnt;
      while (on) {
        const int kt = t0 + __ffs(on) - 1;
        on &= on - 1;
        int32_t di = -1;
        if ((kt + 1) * bn > m.N) {
          tsr_tile_desc d;
          classify(m, bh, h, rs, kt * bn, bn, nqs, nks, &d);
          di = d_pos;
          descs[di] = d;
        }
        entries[at++] = make_int2(kt * bn, di);
      }
      e_pos += __shfl_sync(0xFFFFFFFFu, x, 31);
    }
    return;
  }
  for (int base = 0; base < n_kt; base += 32) {
    const int kt = (base + lane < n_kt) ? kw.tile(base + lane) : 0;
    tsr_tile_desc d;
    const int c = (base + lane < n_kt) ? classify(m, bh, h, rs, kt * bn, bn, nqs, nks, &d) : 0;
    const unsigned nonempty = __ballot_sync(0xFFFFFFFFu, c > 0);
    const unsigned bnd = __ballot_sync(0xFFFFFFFFu, c == 2);
    const unsigned below = (1u << lane) - 1u;
    if (c > 0) {
      const int32_t ei = e_pos + __popc(nonempty & below);
      int32_t di = -1;
      if (c == 2) {
        di = d_pos + __popc(bnd & below);
        descs[di] = d;
      }
      entries[ei] = make_int2(kt * bn, di);
    }
    e_pos += __popc(nonempty);
    d_pos += __popc(bnd);
  }
}

}  // namespace

// Launches of the planner kernels over buffers the caller provides (used by the
// static-scratch entry point; tsr_plan goes through plan_build below).
tsr_status plan_count_into(const MaskDev& m, int32_t nqt, int32_t* cnt, unsigned long long* tot,
                           uint32_t* err, int64_t n_grid, cudaStream_t stream) {
  const int64_t n_items = static_cast<int64_t>(m.B) * m.H * nqt;
  const int threads = 256;
  const int64_t blocks_w = (n_items * 32 + threads - 1) / threads;
  plan_count_kernel<<<static_cast<unsigned>(blocks_w), threads, 0, stream>>>(m, nqt, kBM, cnt, tot,
                                                                             err);
  TSR_CUDA(cudaGetLastError());
  if (n_grid > 0) {
    logical_count_kernel<<<static_cast<unsigned>(std::min<int64_t>(1024, (n_grid + 255) / 256)),
                           256, 0, stream>>>(m.blocks, n_grid, tot + 6);
    TSR_CUDA(cudaGetLastError());
  }
  return TSR_OK;
}

tsr_status plan_finish_into(const MaskDev& m, int32_t nqt, int32_t bn, const int32_t* cnt_e,
                            const int32_t* cnt_b, int32_t max_len, int32_t* ebegin,
                            int32_t* dbegin, int32_t* hist, void* items, void* entries,
                            void* descs, cudaStream_t stream) {
  const int64_t n_items = static_cast<int64_t>(m.B) * m.H * nqt;
  const int threads = 256;
  const int64_t blocks_w = (n_items * 32 + threads - 1) / threads;
  const int32_t all_heads = static_cast<int32_t>(n_items / nqt);
  plan_schedule_kernel<<<1, 1024, schedule_smem(max_len + 1), stream>>>(cnt_e, cnt_b, n_items, nqt, m.H, m.head_kind,
                                               m.kind == TSR_MASK_SVG ? 1 : 0, max_len, 1,
                                               all_heads, max_len + 1, ebegin, dbegin, hist,
                                               static_cast<int4*>(items));
  TSR_CUDA(cudaGetLastError());
  plan_emit_kernel<<<static_cast<unsigned>(blocks_w), threads, 0, stream>>>(
      m, nqt, kBM, bn, ebegin, dbegin, static_cast<int2*>(entries),
      static_cast<tsr_tile_desc*>(descs));
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

tsr_status devbuf_reserve(DevBuf& b, size_t bytes) {
  if (bytes == 0) bytes = 16;
  if (b.cap >= bytes) return TSR_OK;
  cudaFree(b.p);
  b.p = nullptr;
  b.cap = 0;
  const size_t want = bytes + bytes / 4;   // headroom for the next, slightly larger mask
  const cudaError_t e = cudaMalloc(&b.p, want);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(TSR_ERR_OOM, "cudaMalloc of " + std::to_string(want) + " bytes failed");
  }
  b.cap = want;
  return TSR_OK;
}

void devbuf_free(DevBuf& b) {
  cudaFree(b.p);
  b.p = nullptr;
  b.cap = 0;
}

// Heads per scheduling group: as many (b, h) as keep their K and V (2 x N x d
// bf16 each) and the extra bytes per head within ~96 MB of the 126 MB L2.
int32_t heads_per_group(int32_t N, int32_t d, int64_t n_heads, double extra_per_head) {
  const double per_head = 2.0 * N * d * 2.0 + extra_per_head;
  const int64_t g = static_cast<int64_t>(96.0e6 / per_head);
  return static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(g, n_heads)));
}

tsr_status resolve_regime(Regime rg, const tsr_plan_opts* opts, int d, bool gathered,
                          Regime* out) {
  // orientation: the caller's, else 128-row tiles when the caller fixes the
  // pipeline depth or CTAs per SM (parameters of 128-row tiles only), else the
  // table's; key-major tiles exist for d = 128 only (a table row naming them
  // for d = 64 falls back to 128-row tiles)
  int32_t orient = (opts && opts->orient) ? opts->orient
                   : (opts && (opts->stages || opts->ctas_per_sm)) ? TSR_ORIENT_ROWS
                                                                   : rg.orient;
  if (orient != TSR_ORIENT_KEYS) orient = TSR_ORIENT_ROWS;
  if (orient == TSR_ORIENT_KEYS && d != 128) {
    if (opts && opts->orient == TSR_ORIENT_KEYS)
      return fail(TSR_ERR_UNSUPPORTED, "key-major tiles (TSR_ORIENT_KEYS) need d = 128");
    orient = TSR_ORIENT_ROWS;
    if (rg.bn == 0) rg.bn = 64;
  }
  if (orient == TSR_ORIENT_KEYS) {
    // one kernel: 64 x 64 tiles, two per step, fixed rings, one CTA per SM
    if (opts && opts->bn && opts->bn != 64)
      return fail(TSR_ERR_UNSUPPORTED, "key-major tiles are 64 keys wide (bn = 64)");
    *out = Regime{64, 2, 1, (opts && (opts->bn || opts->stages || opts->ctas_per_sm || opts->orient))
                                ? -1 : rg.id, TSR_ORIENT_KEYS};
    return TSR_OK;
  }
  if (opts && (opts->bn || opts->stages || opts->ctas_per_sm)) {
    if (opts->bn && opts->bn != 64 && opts->bn != 128)
      return fail(TSR_ERR_INVALID_ARG, "bn must be 64 or 128");
    int bn = 0, st = 0, ct = 0;
    // the caller's fields, then the table's for the rest if that combination exists
    const int want_bn = opts->bn, want_st = opts->stages, want_ct = opts->ctas_per_sm;
    if (!variant_pick(d, gathered, want_bn ? want_bn : rg.bn, want_st ? want_st : rg.stages,
                      want_ct ? want_ct : rg.ctas, &bn, &st, &ct) &&
        !variant_pick(d, gathered, want_bn, want_st, want_ct, &bn, &st, &ct))
      return fail(TSR_ERR_UNSUPPORTED,
                  "no kernel variant for d=" + std::to_string(d) + " bn=" + std::to_string(want_bn) +
                      " stages=" + std::to_string(want_st) + " ctas=" + std::to_string(want_ct) +
                      (gathered ? " (gathered)" : ""));
    *out = Regime{bn, st, ct, -1, TSR_ORIENT_ROWS};
    return TSR_OK;
  }
  if (!variant_exists(d, rg.bn, rg.stages, rg.ctas, gathered)) {
    int bn = 0, st = 0, ct = 0;
    if (!variant_pick(d, gathered, rg.bn, 0, 0, &bn, &st, &ct) &&
        !variant_pick(d, gathered, 0, 0, 0, &bn, &st, &ct))
      return fail(TSR_ERR_UNSUPPORTED, "no kernel variant for d=" + std::to_string(d));
    *out = Regime{bn, st, ct, rg.id, TSR_ORIENT_ROWS};
    return TSR_OK;
  }
  *out = rg;
  out->orient = TSR_ORIENT_ROWS;
  return TSR_OK;
}

tsr_status plan_schedule_into(const int32_t* cnt_e, const int32_t* cnt_b, int64_t n_items,
                              int32_t nqt, int32_t H, int32_t lpt, int32_t max_len,
                              int32_t group_heads, int32_t* ebegin, int32_t* dbegin,
                              int32_t* hist, void* items, cudaStream_t stream) {
  const int64_t n_groups = (n_items / nqt + group_heads - 1) / group_heads;
  const int64_t n_buckets = n_groups * (max_len + 1);
  plan_schedule_kernel<<<1, 1024, schedule_smem(n_buckets), stream>>>(
      cnt_e, cnt_b, n_items, nqt, H, nullptr, 0, max_len, lpt, group_heads, n_buckets, ebegin,
      dbegin, hist, static_cast<int4*>(items));
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

tsr_status plan_build(const tsr_mask* mask, const tsr_plan_opts* opts, tsr_plan_impl* P,
                      cudaStream_t stream) {
  const int32_t B = mask->B, H = mask->H, N = mask->N;
  MaskDev m;
  memset(&m, 0, sizeof m);
  m.kind = mask->kind;
  m.B = B;
  m.H = H;
  m.N = N;
  m.bq = mask->bq;
  m.bk = mask->bk;
  m.n_qseg = mask->n_qseg;
  m.n_kseg = mask->n_kseg;
  m.q_bounds = mask->q_bounds;
  m.k_bounds = mask->k_bounds;
  m.blocks = mask->blocks;
  m.F = mask->n_frames;
  m.S = mask->frame_size;
  m.R = mask->temporal_radius;
  m.head_kind = P->head_kind_dev;

  if (tsr_status s = devbuf_reserve(P->b_tot, sizeof(unsigned long long) * 8)) return s;
  if (!P->host_tot) TSR_CUDA(cudaMallocHost(&P->host_tot, sizeof(unsigned long long) * 9));
  unsigned long long* tot = static_cast<unsigned long long*>(P->b_tot.p);
  unsigned long long* host_tot = P->host_tot;
  TSR_CUDA(cudaMemsetAsync(tot, 0, sizeof(unsigned long long) * 8, stream));
  TSR_CUDA(cudaMemsetAsync(P->err, 0, sizeof(uint32_t), stream));

  // 1. the mask's density for the regime table (logical blocks counted on the
  // GPU; SVG from the head kinds, whose host copy was queued by the caller)
  int64_t n_grid = 0;
  if (m.kind == TSR_MASK_UNIFORM) {
    n_grid = static_cast<int64_t>(B) * H * ((N + m.bq - 1) / m.bq) * ((N + m.bk - 1) / m.bk);
  } else if (m.kind == TSR_MASK_SEGMENTS) {
    n_grid = static_cast<int64_t>(B) * H * m.n_qseg * m.n_kseg;
  }
  if (n_grid > 0) {
    logical_count_kernel<<<static_cast<unsigned>(std::min<int64_t>(1024, (n_grid + 255) / 256)),
                           256, 0, stream>>>(m.blocks, n_grid, tot + 6);
    TSR_CUDA(cudaGetLastError());
    TSR_CUDA(cudaMemcpyAsync(host_tot + 6, tot + 6, sizeof(unsigned long long),
                             cudaMemcpyDeviceToHost, stream));
  }
  // A re-plan usually keeps its regime: the tiles are counted at the previous
  // plan's tile height before the regime is known, and their totals come back
  // with the density, so a plan whose height is unchanged synchronises once.
  int32_t spec_bm = (P->n_items > 0 && (P->bm == 64 || P->bm == kBM)) ? P->bm : 0;
  if (spec_bm && static_cast<int64_t>(B) * H * ((N + spec_bm - 1) / spec_bm) > (int64_t{1} << 30))
    spec_bm = 0;                                   // too many tiles at that height: no guess
  const int threads = 256;
  auto count_tiles = [&](int32_t bm_c) -> tsr_status {
    const int32_t nqt_c = (N + bm_c - 1) / bm_c;
    const int64_t n_items_c = static_cast<int64_t>(B) * H * nqt_c;
    if (n_items_c > (int64_t{1} << 30)) return fail(TSR_ERR_UNSUPPORTED, "too many query tiles");
    if (tsr_status s = devbuf_reserve(P->b_cnt, sizeof(int32_t) * 4 * n_items_c)) return s;
    const int64_t blocks_c = (n_items_c * 32 + threads - 1) / threads;
    plan_count_kernel<<<static_cast<unsigned>(blocks_c), threads, 0, stream>>>(
        m, nqt_c, bm_c, static_cast<int32_t*>(P->b_cnt.p), tot, P->err);
    TSR_CUDA(cudaGetLastError());
    TSR_CUDA(cudaMemcpyAsync(host_tot, tot, sizeof(unsigned long long) * 6, cudaMemcpyDeviceToHost,
                             stream));
    TSR_CUDA(cudaMemcpyAsync(host_tot + 8, P->err, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream));
    return TSR_OK;
  };
  if (spec_bm)
    if (tsr_status s = count_tiles(spec_bm)) return s;
  TSR_CUDA(cudaStreamSynchronize(stream));
  if (m.kind == TSR_MASK_SVG) {
    for (int32_t h = 0; h < H; ++h) {
      const int8_t k = P->host_kinds[h];
      if (k != TSR_HEAD_SPATIAL && k != TSR_HEAD_TEMPORAL)
        return fail(TSR_ERR_INVALID_ARG, "head_kind values must be 0 or 1");
      P->head_layout[h] = k;
      P->n_temporal += k;
    }
  }
  double density = 0.0;
  if (n_grid > 0) {
    P->n_logical_on = static_cast<int64_t>(host_tot[6]);
    P->n_logical_total = n_grid;
    density = static_cast<double>(host_tot[6]) / static_cast<double>(n_grid);
  } else if (m.kind == TSR_MASK_SVG) {
    // allowed elements per head: spatial S^2 (2F - 1); temporal with radius r
    // F^2 (S (2r + 1) - r (r + 1)) while r < S, else N^2
    const double S = m.S, F = m.F, r = m.R;
    const double temporal = (m.R < m.S) ? F * F * (S * (2 * r + 1) - r * (r + 1))
                                        : static_cast<double>(N) * N;
    double on = 0;
    for (int32_t h = 0; h < H; ++h) on += (P->head_layout[h] ? temporal : S * S * (2 * F - 1));
    P->n_logical_on = static_cast<int64_t>(on) * B;
    P->n_logical_total = static_cast<int64_t>(B) * H * N * static_cast<int64_t>(N);
    density = on / (static_cast<double>(H) * N * static_cast<double>(N));
  }

  // 2. the regime: tile orientation (query rows per tile), width, pipeline
  Regime rg;
  if (tsr_status s = resolve_regime(regime_lookup(m.kind, m.bq, m.bk, N, density, P->d), opts,
                                    P->d, false, &rg))
    return s;
  P->bn = rg.bn;
  P->stages = rg.stages;
  P->ctas = rg.ctas;
  P->regime_id = rg.id;
  P->orient = rg.orient;
  P->bm = bm_of(rg.orient);
  const int32_t bm = P->bm;
  const int32_t nqt = (N + bm - 1) / bm;
  const int64_t n_items = static_cast<int64_t>(B) * H * nqt;
  P->n_items = n_items;
  if (n_items > (int64_t{1} << 30)) return fail(TSR_ERR_UNSUPPORTED, "too many query tiles");

  // 3. tiles per query tile (both widths at the chosen height), unless the
  // speculative count above was at this height
  if (bm != spec_bm) {
    if (spec_bm) {
      // the speculative totals and error bits belong to another height
      TSR_CUDA(cudaMemsetAsync(tot, 0, sizeof(unsigned long long) * 6, stream));
      TSR_CUDA(cudaMemsetAsync(P->err, 0, sizeof(uint32_t), stream));
    }
    if (tsr_status s = count_tiles(bm)) return s;
    TSR_CUDA(cudaStreamSynchronize(stream));
  }
  int32_t* cnt = static_cast<int32_t*>(P->b_cnt.p);
  const int64_t blocks_w = (n_items * 32 + threads - 1) / threads;
  const uint32_t host_err = static_cast<uint32_t>(host_tot[8] & 0xFFFFFFFFull);
  if (host_err & DEV_ERR_UNSUPPORTED)
    return fail(TSR_ERR_UNSUPPORTED,
                "a " + std::to_string(bm) + "-token tile overlaps more than 8 logical segments "
                "(blocks or segments smaller than 16 tokens)");
  if (host_err) return fail(TSR_ERR_INTERNAL, "planner error word " + std::to_string(host_err));
  const int which = (rg.bn == 64) ? 0 : 1;
  P->n_entries = static_cast<int64_t>(host_tot[2 * which]);
  P->n_desc = static_cast<int64_t>(host_tot[2 * which + 1]);
  P->max_item_len = static_cast<int64_t>(host_tot[4 + which]);
  if (P->n_entries >= (int64_t{1} << 31) || P->n_desc >= (int64_t{1} << 31))
    return fail(TSR_ERR_UNSUPPORTED, "plan has more than 2^31 tiles");

  // 4. longest-first schedule and the tiles themselves
  if (tsr_status s = devbuf_reserve(P->b_items, sizeof(tsr_plan_item) * n_items)) return s;
  if (tsr_status s = devbuf_reserve(P->b_entries, sizeof(tsr_plan_entry) * P->n_entries)) return s;
  if (tsr_status s = devbuf_reserve(P->b_descs, sizeof(tsr_tile_desc) * P->n_desc)) return s;
  if (tsr_status s = devbuf_reserve(P->b_ebegin, sizeof(int32_t) * n_items)) return s;
  if (tsr_status s = devbuf_reserve(P->b_dbegin, sizeof(int32_t) * n_items)) return s;
  const int32_t group_heads = P->group_heads > 0 ? P->group_heads
                                                 : heads_per_group(N, P->d, static_cast<int64_t>(B) * H);
  const int64_t n_groups = (static_cast<int64_t>(B) * H + group_heads - 1) / group_heads;
  const int64_t n_buckets = n_groups * (P->max_item_len + 1);
  if (tsr_status s = devbuf_reserve(P->b_hist, sizeof(int32_t) * (n_buckets + 1))) return s;
  P->items = P->b_items.p;
  P->entries = P->b_entries.p;
  P->descs = P->b_descs.p;
  int32_t* ebegin = static_cast<int32_t*>(P->b_ebegin.p);
  int32_t* dbegin = static_cast<int32_t*>(P->b_dbegin.p);
  int32_t* hist = static_cast<int32_t*>(P->b_hist.p);
  const int32_t* cnt_e = cnt + (2 * which) * n_items;
  const int32_t* cnt_b = cnt + (2 * which + 1) * n_items;
  const int lpt = (opts && (opts->flags & TSR_PLAN_NO_LPT)) ? 0 : 1;
  plan_schedule_kernel<<<1, 1024, schedule_smem(n_buckets), stream>>>(
      cnt_e, cnt_b, n_items, nqt, H, P->head_kind_dev, m.kind == TSR_MASK_SVG ? 1 : 0,
      static_cast<int32_t>(P->max_item_len), lpt, group_heads, n_buckets, ebegin, dbegin, hist,
      static_cast<int4*>(P->items));
  TSR_CUDA(cudaGetLastError());
  plan_emit_kernel<<<static_cast<unsigned>(blocks_w), threads, 0, stream>>>(
      m, nqt, bm, rg.bn, ebegin, dbegin, static_cast<int2*>(P->entries),
      static_cast<tsr_tile_desc*>(P->descs));
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

// --------------------------------------------------------- launch list (SVG)
//
// Sparse VideoGen digest, "Sparse VideoGen": with radius 0 a temporal head's
// allowed pairs are the F x F blocks of the tokens at one spatial position, too
// small for 64- or 128-row tiles.  svg_temporal.cu computes them; the attention
// kernels take the spatial heads' items, in the order the scheduler gave them.
namespace {

// Stable compaction of the items whose head is not temporal, by one CTA: each
// thread takes a contiguous run of items, the runs' kept counts are scanned.
// The head kinds sit in shared memory (up to kCompactMaxH heads) and each
// thread's item loads are issued four at a time.
constexpr int32_t kCompactMaxH = 4096;

__global__ void __launch_bounds__(1024) launch_compact_kernel(const int4* items, int64_t n_items,
                                                              const int8_t* head_kind, int32_t H,
                                                              int4* launch) {
  __shared__ int64_t warp_sum[32];
  __shared__ int8_t kinds[kCompactMaxH];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, n_warps = blockDim.x >> 5;
  const bool shared_kinds = H <= kCompactMaxH;
  if (shared_kinds)
    for (int h = t; h < H; h += blockDim.x) kinds[h] = head_kind[h];
  __syncthreads();
  auto temporal = [&](int32_t bh) {
    const int32_t h = bh % H;
    return (shared_kinds ? kinds[h] : head_kind[h]) == TSR_HEAD_TEMPORAL;
  };
  constexpr int kBatch = 4;
  const int64_t per = (n_items + blockDim.x - 1) / blockDim.x;
  const int64_t i0 = min(n_items, t * per), i1 = min(n_items, i0 + per);
  int64_t kept = 0;
  for (int64_t b = i0; b < i1; b += kBatch) {
    int32_t bh[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) bh[j] = b + j < i1 ? items[2 * (b + j)].x : 0;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) kept += (b + j < i1 && !temporal(bh[j])) ? 1 : 0;
  }
  int64_t x = kept;                                       // inclusive scan in the warp
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < n_warps ? warp_sum[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    warp_sum[lane] = w;
  }
  __syncthreads();
  int64_t at = x - kept + (warp ? warp_sum[warp - 1] : 0);
  for (int64_t b = i0; b < i1; b += kBatch) {
    int4 a[kBatch], c[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const bool ok = b + j < i1;
      a[j] = ok ? items[2 * (b + j)] : make_int4(0, 0, 0, 0);
      c[j] = ok ? items[2 * (b + j) + 1] : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      if (b + j < i1 && !temporal(a[j].x)) {
        launch[2 * at] = a[j];
        launch[2 * at + 1] = c[j];
        ++at;
      }
    }
  }
}

}  // namespace

tsr_status plan_launch_list(tsr_plan_impl* P, cudaStream_t stream) {
  const int64_t BH = static_cast<int64_t>(P->B) * P->H;
  P->temporal_band = 0;
  P->launch = P->items;
  P->n_launch = P->n_items;
  P->spatial_before.clear();
  if (P->kind != TSR_MASK_SVG || P->n_temporal == 0 || !svg_temporal_eligible(P->F, P->R, P->d) ||
      (P->flags & (TSR_PLAN_DEBUG_CHECKS | TSR_PLAN_TEMPORAL_TILES)))
    return TSR_OK;
  P->spatial_before.assign(BH + 1, 0);
  for (int64_t bh = 0; bh < BH; ++bh)
    P->spatial_before[bh + 1] = P->spatial_before[bh] + (P->head_layout[bh % P->H] ? 0 : 1);
  const int64_t nqt = (P->N + P->bm - 1) / P->bm;   // every head has nqt items
  if (!P->band_stream) TSR_CUDA(cudaStreamCreateWithFlags(&P->band_stream, cudaStreamNonBlocking));
  if (!P->band_fork) TSR_CUDA(cudaEventCreateWithFlags(&P->band_fork, cudaEventDisableTiming));
  if (!P->band_join) TSR_CUDA(cudaEventCreateWithFlags(&P->band_join, cudaEventDisableTiming));
  P->temporal_band = 1;
  P->n_launch = nqt * P->spatial_before[BH];
  if (P->n_launch == 0) return TSR_OK;
  if (tsr_status st = devbuf_reserve(P->b_launch, sizeof(tsr_plan_item) * P->n_launch)) return st;
  P->launch = P->b_launch.p;
  launch_compact_kernel<<<1, 1024, 0, stream>>>(static_cast<const int4*>(P->items), P->n_items,
                                                 P->head_kind_dev, P->H, static_cast<int4*>(P->launch));
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

// ------------------------------------------------------------------ split-KV
//
// Tessera abstract: task organisation exposes parallelism.  A request with few
// work items (a few heads) leaves CTA slots idle while its last items run; the
// split plan cuts each item's tile list [begin, end) into kv_split contiguous
// parts of near-equal length (key-major plans cut on whole steps of two tiles).
// The items cut are those of the launch list (without the SVG temporal heads
// that run on their own kernel); i below indexes that list.
// Part p of item i is work unit i * kv_split + p: units keep the items'
// longest-first order, and the units of one head stay one contiguous range.
// A unit's second int4 carries (layout, i, kv_split, p); the attention kernel
// writes the unit's normalised partial O and lse, and the last unit of an item
// to finish merges the parts:  lse = log2 sum_p 2^lse_p,
// O = sum_p 2^(lse_p - lse) O_p  (all parts empty: O = 0, lse = -inf).
namespace {

__global__ void split_units_kernel(const int4* items, int64_t n_items, int32_t s, int32_t step,
                                   int4* units) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_items) return;
  const int4 a = items[2 * i], b = items[2 * i + 1];
  const int32_t n = a.w - a.z;
  const int32_t steps = (n + step - 1) / step;       // whole steps of `step` tiles
  for (int32_t p = 0; p < s; ++p) {
    const int32_t c0 = min(n, step * static_cast<int32_t>((static_cast<int64_t>(p) * steps) / s));
    const int32_t c1 = min(n, step * static_cast<int32_t>((static_cast<int64_t>(p + 1) * steps) / s));
    const int64_t u = i * s + p;
    units[2 * u] = make_int4(a.x, a.y, a.z + c0, a.z + c1);
    units[2 * u + 1] = make_int4(b.x, static_cast<int32_t>(i), s, p);
  }
}

}  // namespace

tsr_status plan_split(tsr_plan_impl* P, const tsr_plan_opts* opts, cudaStream_t stream) {
  int32_t s = 1;
  if (opts && opts->kv_split) {
    s = opts->kv_split;
  } else {
    // 128-row plans with fewer work items than CTA slots leave CTAs without
    // work: cut the items until every slot has one (one 8,192-token head: 64
    // items on 304 slots, 52 -> 31 us).  With more items than slots a split
    // costs more than the tail it removes (each part pays the per-item
    // pipeline start, the partial-result traffic and the merge), and so it
    // does for key-major plans, whose items are 64 rows already (one
    // 8,192-token head, 128 items on 152 slots: 24 -> 37 us).
    if (P->orient != TSR_ORIENT_KEYS) {
      const int64_t slots = static_cast<int64_t>(num_sms(P->device)) * P->ctas;
      while (s < 4 && P->n_launch * s < slots) s *= 2;
    }
  }
  P->kv_split = s;
  P->units = nullptr;
  if (s == 1 || P->n_launch == 0) {
    P->kv_split = 1;
    return TSR_OK;
  }
  const int64_t n_units = P->n_launch * s;
  if (n_units >= (int64_t{1} << 31)) return fail(TSR_ERR_UNSUPPORTED, "too many split-KV work units");
  const size_t rows = static_cast<size_t>(n_units) * P->bm;
  if (tsr_status st = devbuf_reserve(P->b_units, sizeof(tsr_plan_item) * n_units)) return st;
  if (tsr_status st = devbuf_reserve(P->b_part_o, rows * P->d * sizeof(float))) return st;
  if (tsr_status st = devbuf_reserve(P->b_part_lse, rows * sizeof(float))) return st;
  if (tsr_status st = devbuf_reserve(P->b_part_cnt, sizeof(int32_t) * P->n_launch)) return st;
  P->units = P->b_units.p;
  const int threads = 256;
  split_units_kernel<<<static_cast<unsigned>((P->n_launch + threads - 1) / threads), threads, 0, stream>>>(
      static_cast<const int4*>(P->launch), P->n_launch, s, P->orient == TSR_ORIENT_KEYS ? 2 : 1,
      static_cast<int4*>(P->units));
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

}  // namespace tsr
