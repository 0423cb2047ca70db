// plan_keylist.cu -- planning of M x 1 key-slice (KEYLIST) masks.
//
// FG-Attn abstract: attention is skipped at the granularity of M x 1 slices (a
// block of M = 64 queries times one key); for each query block only its listed
// keys are loaded, gathered into packed tiles in shared memory.  Physical tiles
// are 128 query rows, so a query tile holds two 64-query blocks (or one block
// when M = 128).  The tile's key stream is the sorted union of its blocks'
// lists, cut into BN-key gathered tiles; each gathered tile carries the key
// indices (gidx) and a list descriptor with one BN-bit column mask per query
// block (a key of the union that one block does not list is masked for that
// block's rows).  Tiles where both blocks list every key are marked full.
//
// Kernels: validate (lists sorted, unique, in range), count (union sizes for
// both tile widths), the shared schedule kernel (longest first), emit (one
// block per query tile merges the two lists).
#include <algorithm>
#include <climits>
#include <cstring>
#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace tsr {

namespace {

__device__ __forceinline__ int64_t lower_bound_i32(const int32_t* a, int64_t n, int32_t x) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// One warp per list.
__global__ void keylist_validate_kernel(const int64_t* indptr, const int32_t* indices,
                                        int64_t n_lists, int32_t N, uint32_t* err) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= n_lists) return;
  const int64_t b = indptr[w], e = indptr[w + 1];
  bool bad = (w == 0 && b != 0) || e < b;
  if (!bad) {
    for (int64_t q = b + lane; q < e; q += 32) {
      const int32_t k = indices[q];
      if (k < 0 || k >= N || (q + 1 < e && indices[q + 1] <= k)) bad = true;
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(err, DEV_ERR_BAD_INPUT);
}

struct Lists {
  const int32_t* a;
  const int32_t* b;
  int64_t na, nb;
  bool b_rows;   // rows of the second block exist (inside [0, N))
};

__device__ __forceinline__ Lists tile_lists(const int64_t* indptr, const int32_t* indices,
                                            int64_t item, int32_t nqt, int32_t nqb, int32_t slice_m,
                                            int32_t N) {
  const int64_t bh = item / nqt, qt = item % nqt;
  Lists L;
  const int64_t qa = (slice_m == 64) ? 2 * qt : qt;
  const int64_t ra = bh * nqb + qa;
  L.a = indices + indptr[ra];
  L.na = indptr[ra + 1] - indptr[ra];
  L.b = L.a;
  L.nb = 0;
  L.b_rows = false;
  if (slice_m == 64 && qa + 1 < nqb) {
    L.b = indices + indptr[ra + 1];
    L.nb = indptr[ra + 2] - indptr[ra + 1];
    L.b_rows = true;
  }
  return L;
}

// Per query tile: [0] tiles at BN=64, [1] tiles at BN=128, [2] union size.
// Totals: [0] tiles BN=64, [1] tiles BN=128, [2] max BN=64, [3] max BN=128,
// [4] sum of list lengths.
__global__ void keylist_count_kernel(const int64_t* indptr, const int32_t* indices, int64_t n_items,
                                     int32_t nqt, int32_t nqb, int32_t slice_m, int32_t N,
                                     int32_t* cnt, unsigned long long* tot) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= n_items) return;
  const Lists L = tile_lists(indptr, indices, w, nqt, nqb, slice_m, N);
  // common keys: search the shorter list's keys in the longer one
  const int32_t* s = L.na <= L.nb ? L.a : L.b;
  const int32_t* g = L.na <= L.nb ? L.b : L.a;
  const int64_t ns = L.na <= L.nb ? L.na : L.nb, ng = L.na <= L.nb ? L.nb : L.na;
  int64_t common = 0;
  for (int64_t i = lane; i < ns; i += 32) {
    const int64_t k = lower_bound_i32(g, ng, s[i]);
    common += (k < ng && g[k] == s[i]);
  }
  for (int o = 16; o > 0; o >>= 1) common += __shfl_xor_sync(0xFFFFFFFFu, common, o);
  if (lane == 0) {
    const int64_t u = L.na + L.nb - common;
    const int32_t e64 = static_cast<int32_t>((u + 63) / 64), e128 = static_cast<int32_t>((u + 127) / 128);
    cnt[w] = e64;
    cnt[n_items + w] = e128;
    cnt[2 * n_items + w] = static_cast<int32_t>(u);
    atomicAdd(&tot[0], static_cast<unsigned long long>(e64));
    atomicAdd(&tot[1], static_cast<unsigned long long>(e128));
    atomicMax(&tot[2], static_cast<unsigned long long>(e64));
    atomicMax(&tot[3], static_cast<unsigned long long>(e128));
    atomicAdd(&tot[4], static_cast<unsigned long long>(L.na + L.nb));
  }
}

// Exclusive prefix sum of one flag per thread over the block (blockDim = 256);
// returns this thread's prefix and adds the block total to *carry (uniform).
__device__ __forceinline__ int block_scan_flags(int flag, int* warp_tot, int* carry) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xFFFFFFFFu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(bal);
  __syncthreads();
  int before = 0, total = 0;
  for (int i = 0; i < 8; ++i) {
    const int t = warp_tot[i];
    if (i < warp) before += t;
    total += t;
  }
  const int res = *carry + before + in_warp;
  __syncthreads();
  if (threadIdx.x == 0) *carry += total;
  __syncthreads();
  return res;
}

// One block of 256 threads per query tile: merge the two sorted lists into the
// union, write each union key at its rank into gidx, set its column bit for the
// block(s) that list it, pad the last tile, then mark full tiles.
__global__ void __launch_bounds__(256) keylist_emit_kernel(
    const int64_t* indptr, const int32_t* indices, int32_t nqt, int32_t nqb, int32_t slice_m,
    int32_t N, int32_t bn, const int32_t* cnt_e, const int32_t* cnt_u, const int32_t* ebegin,
    int2* entries, uint32_t* descs, int32_t* gidx) {
  __shared__ int warp_tot[8];
  __shared__ int carry;
  const int64_t item = blockIdx.x;
  const Lists L = tile_lists(indptr, indices, item, nqt, nqb, slice_m, N);
  const int64_t e0 = ebegin[item];
  const int32_t ne = cnt_e[item];
  const int64_t u = cnt_u[item];
  uint32_t* dw = descs + e0 * 8;                 // 8 words (32 bytes) per tile
  for (int64_t i = threadIdx.x; i < static_cast<int64_t>(ne) * 8; i += blockDim.x) dw[i] = 0u;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  int32_t* gx = gidx + e0 * bn;
  // keys of the first list: rank = i + #{b < a} - #{common keys before a}
  for (int64_t base = 0; base < L.na; base += blockDim.x) {
    const int64_t i = base + threadIdx.x;
    int32_t a = 0;
    int64_t lb = 0;
    int in_b = 0;
    if (i < L.na) {
      a = L.a[i];
      lb = lower_bound_i32(L.b, L.nb, a);
      in_b = (lb < L.nb && L.b[lb] == a);
    }
    const int common_before = block_scan_flags(in_b, warp_tot, &carry);
    if (i < L.na) {
      const int64_t pos = i + lb - common_before;
      gx[pos] = a;
      uint32_t* d = dw + (pos / bn) * 8;
      const int c = static_cast<int>(pos % bn);
      atomicOr(&d[c >> 5], 1u << (c & 31));
      if (in_b) atomicOr(&d[4 + (c >> 5)], 1u << (c & 31));
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  // keys only the second list holds: rank = j + #{a < b} - #{common keys before b}
  for (int64_t base = 0; base < L.nb; base += blockDim.x) {
    const int64_t j = base + threadIdx.x;
    int32_t b = 0;
    int64_t lb = 0;
    int in_a = 0;
    if (j < L.nb) {
      b = L.b[j];
      lb = lower_bound_i32(L.a, L.na, b);
      in_a = (lb < L.na && L.a[lb] == b);
    }
    const int common_before = block_scan_flags(in_a, warp_tot, &carry);
    if (j < L.nb && !in_a) {
      const int64_t pos = j + lb - common_before;
      gx[pos] = b;
      uint32_t* d = dw + (pos / bn) * 8;
      const int c = static_cast<int>(pos % bn);
      atomicOr(&d[4 + (c >> 5)], 1u << (c & 31));
    }
  }
  // padding of the last tile: any in-range key; its columns stay masked
  for (int64_t pos = u + threadIdx.x; pos < static_cast<int64_t>(ne) * bn; pos += blockDim.x)
    gx[pos] = 0;
  __threadfence_block();
  __syncthreads();
  for (int32_t c = threadIdx.x; c < ne; c += blockDim.x) {
    const volatile uint32_t* d = dw + c * 8;
    bool full = static_cast<int64_t>(c + 1) * bn <= u;
    for (int w = 0; w < bn / 32; ++w) {
      full = full && d[w] == 0xFFFFFFFFu;
      if (L.b_rows) full = full && d[4 + w] == 0xFFFFFFFFu;
    }
    entries[e0 + c] = make_int2(static_cast<int32_t>((e0 + c) * bn),
                                full ? -1 : static_cast<int32_t>(e0 + c));
  }
}

// Bitmap form (N up to kBitmapMaxN): one block per query tile builds the two
// lists' key bitmaps in shared memory; union ranks are popcount prefixes, so no
// searching is needed.
constexpr int32_t kBitmapMaxN = 196608;

__host__ __device__ constexpr int32_t bitmap_words(int32_t N) { return (N + 31) >> 5; }
// one bitmap's words rounded up to 16 bytes (the second bitmap starts aligned)
__host__ __device__ constexpr int32_t bitmap_words16(int32_t N) { return (bitmap_words(N) + 3) & ~3; }

// One shared atomic per run of a thread's keys that share a bitmap word.
__device__ __forceinline__ void or_keys4(uint32_t* bm, int4 v) {
  uint32_t w = static_cast<uint32_t>(v.x) >> 5, bits = 1u << (v.x & 31);
  const int32_t rest[3] = {v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint32_t wj = static_cast<uint32_t>(rest[j]) >> 5;
    if (wj != w) {
      atomicOr(&bm[w], bits);
      w = wj;
      bits = 0u;
    }
    bits |= 1u << (rest[j] & 31);
  }
  atomicOr(&bm[w], bits);
}

// Sets one bit per key of a sorted list in a shared bitmap (all threads of the
// block take part).  The list is read with 16-byte loads, four per thread in
// flight: scalar keys up to the first 16-byte boundary, then whole vectors,
// then a scalar tail.  With CHECK, a key outside [0, N) or not above its
// predecessor is reported (return value) and its vector is not set; without it
// the list must already be known to be valid.
template <bool CHECK>
__device__ bool set_bits_vec(uint32_t* bm, const int32_t* keys, int64_t n, int32_t N) {
  bool bad = false;
  const int lane = threadIdx.x & 31;
  const int64_t head =
      min(n, static_cast<int64_t>(((16u - (reinterpret_cast<uintptr_t>(keys) & 15u)) & 15u) >> 2));
  const int64_t n4 = (n - head) >> 2;
  auto scalar = [&](int64_t i) {
    const int32_t k = keys[i];
    if (CHECK && (k < 0 || k >= N || (i + 1 < n && keys[i + 1] <= k))) {
      bad = true;
      return;
    }
    atomicOr(&bm[static_cast<uint32_t>(k) >> 5], 1u << (k & 31));
  };
  if (threadIdx.x < head) scalar(threadIdx.x);
  const int4* v4 = reinterpret_cast<const int4*>(keys + head);
  const int64_t T = blockDim.x;
  for (int64_t base = 0; base < n4; base += 4 * T) {
    int4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = base + u * T + threadIdx.x;
      v[u] = i < n4 ? __ldg(v4 + i) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = base + u * T + threadIdx.x;
      if (CHECK) {
        // the key after this vector: the next lane's first key, else a load
        int32_t nx = __shfl_down_sync(0xFFFFFFFFu, v[u].x, 1);
        if (lane == 31 || i + 1 >= n4) {
          const int64_t after = head + 4 * i + 4;
          nx = (i < n4 && after < n) ? keys[after] : INT32_MAX;
        }
        if (i < n4) {
          const int4 k = v[u];
          if (k.x < 0 || k.w >= N || k.y <= k.x || k.z <= k.y || k.w <= k.z || nx <= k.w) {
            bad = true;
            continue;
          }
        }
      }
      if (i < n4) or_keys4(bm, v[u]);
    }
  }
  const int64_t t0 = head + 4 * n4;
  if (threadIdx.x < n - t0) scalar(t0 + threadIdx.x);
  return bad;
}

// Count (bitmap form), validating the tile's lists on the way: indptr must run
// upward from 0 and each list must be ascending, unique and inside [0, N).  A
// bad list sets DEV_ERR_BAD_INPUT and is not used as an index; the host checks
// the error word before anything reads the counts.  Every list belongs to
// exactly one query tile, so every list is checked once.
__device__ __forceinline__ bool list_ok(const int64_t* indptr, int64_t row) {
  return indptr[row + 1] >= indptr[row] && (row != 0 || indptr[0] == 0);
}

__global__ void __launch_bounds__(256) keylist_count_bitmap_kernel(
    const int64_t* indptr, const int32_t* indices, int64_t n_items, int32_t nqt, int32_t nqb,
    int32_t slice_m, int32_t N, int32_t* cnt, unsigned long long* tot, uint32_t* err) {
  extern __shared__ __align__(16) uint32_t sm[];
  __shared__ int wsum[8];
  const int32_t nw = bitmap_words(N), nw16 = bitmap_words16(N);
  uint32_t* bma = sm;
  uint32_t* bmb = sm + nw16;
  const int64_t item = blockIdx.x;
  const int64_t bh = item / nqt, qt = item % nqt;
  const int64_t qa = (slice_m == 64) ? 2 * qt : qt;
  const int64_t ra = bh * nqb + qa;
  const bool two = slice_m == 64 && qa + 1 < nqb;
  if (!list_ok(indptr, ra) || (two && !list_ok(indptr, ra + 1))) {
    if (threadIdx.x == 0) atomicOr(err, DEV_ERR_BAD_INPUT);
    return;
  }
  const Lists L = tile_lists(indptr, indices, item, nqt, nqb, slice_m, N);
  for (int w = threadIdx.x; w < 2 * nw16; w += blockDim.x) sm[w] = 0u;
  __syncthreads();
  bool bad = set_bits_vec<true>(bma, L.a, L.na, N);
  bad = set_bits_vec<true>(bmb, L.b, L.nb, N) || bad;
  if (bad) atomicOr(err, DEV_ERR_BAD_INPUT);
  __syncthreads();
  int s = 0;
  for (int w = threadIdx.x; w < nw; w += blockDim.x) s += __popc(bma[w] | bmb[w]);
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t u = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) u += wsum[i];
    const int32_t e64 = static_cast<int32_t>((u + 63) / 64), e128 = static_cast<int32_t>((u + 127) / 128);
    cnt[item] = e64;
    cnt[n_items + item] = e128;
    cnt[2 * n_items + item] = static_cast<int32_t>(u);
    atomicAdd(&tot[0], static_cast<unsigned long long>(e64));
    atomicAdd(&tot[1], static_cast<unsigned long long>(e128));
    atomicMax(&tot[2], static_cast<unsigned long long>(e64));
    atomicMax(&tot[3], static_cast<unsigned long long>(e128));
    atomicAdd(&tot[4], static_cast<unsigned long long>(L.na + L.nb));
  }
}

// The emit kernel runs 8 warps; each stages the union keys of one 32-word
// chunk of the bitmaps (at most 1024) before writing them out in rank order.
constexpr int kEmitWarps = 8;
constexpr int kStageKeys = 1024;

// Shared memory of the bitmap emit kernel, in 32-bit words: the two lists' key
// bitmaps, the two membership masks in union-rank order (8 words of slack: the
// last tile's mask words may reach past the union), and the warps' stages.
__host__ __device__ constexpr size_t emit_bitmap_words(int32_t N) {
  return 2 * static_cast<size_t>(bitmap_words16(N)) + 2 * static_cast<size_t>(bitmap_words(N) + 8) +
         static_cast<size_t>(kEmitWarps) * kStageKeys;
}

// One block per query tile.  Warp w owns a contiguous range of 32-word chunks
// of the bitmaps; a first pass counts the union keys of each warp's range (the
// block scan of those counts gives each warp its first rank), the second walks
// the chunks in order: a warp scan of the words' popcounts places each word's
// keys in the warp's stage, and the stage goes out to gidx in 32-aligned rank
// groups, whose membership bits are one ballot per list.
__global__ void __launch_bounds__(256) keylist_emit_bitmap_kernel(
    const int64_t* indptr, const int32_t* indices, int32_t nqt, int32_t nqb, int32_t slice_m,
    int32_t N, int32_t bn, const int32_t* cnt_e, const int32_t* ebegin, int2* entries,
    uint32_t* descs, int32_t* gidx) {
  extern __shared__ __align__(16) uint32_t sm[];
  __shared__ int wtot[kEmitWarps];
  const int32_t nw = bitmap_words(N), nw16 = bitmap_words16(N);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t* bma = sm;
  uint32_t* bmb = sm + nw16;
  uint32_t* rka = sm + 2 * nw16;                 // membership of list a, union-rank order
  uint32_t* rkb = rka + nw + 8;                  // membership of list b
  uint32_t* stage = rkb + nw + 8 + warp * kStageKeys;
  const int64_t item = blockIdx.x;
  const Lists L = tile_lists(indptr, indices, item, nqt, nqb, slice_m, N);
  const int64_t e0 = ebegin[item];
  const int32_t ne = cnt_e[item];
  for (int w = threadIdx.x; w < 2 * nw16 + 2 * (nw + 8); w += blockDim.x) sm[w] = 0u;
  __syncthreads();
  set_bits_vec<false>(bma, L.a, L.na, N);
  set_bits_vec<false>(bmb, L.b, L.nb, N);
  __syncthreads();
  const int32_t nch = (nw + 31) >> 5, cpw = (nch + kEmitWarps - 1) / kEmitWarps;
  const int32_t c0 = warp * cpw, c1 = min(nch, c0 + cpw);
  int cnt = 0;
  for (int32_t c = c0; c < c1; ++c) {
    const int32_t w = c * 32 + lane;
    if (w < nw) cnt += __popc(bma[w] | bmb[w]);
  }
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
  if (lane == 0) wtot[warp] = cnt;
  __syncthreads();
  int32_t rank = 0, u = 0;
  for (int i = 0; i < kEmitWarps; ++i) {
    if (i < warp) rank += wtot[i];
    u += wtot[i];
  }
  int32_t* gx = gidx + e0 * bn;
  uint32_t* dw = descs + e0 * 8;
  for (int32_t c = c0; c < c1; ++c) {
    const int32_t w = c * 32 + lane;
    const uint32_t A = w < nw ? bma[w] : 0u, Bm = w < nw ? bmb[w] : 0u;
    uint32_t bits = A | Bm;
    const int x = __popc(bits);
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const int ctot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    // keys are below 2^30: bits 30 and 31 carry membership in a and b
    int k = incl - x;
    while (bits) {
      const int bit = __ffs(bits) - 1;
      bits &= bits - 1u;
      stage[k++] = (static_cast<uint32_t>(w) << 5 | static_cast<uint32_t>(bit)) |
                   ((A >> bit) & 1u) << 30 | ((Bm >> bit) & 1u) << 31;
    }
    __syncwarp();
    for (int32_t p0 = rank & ~31; p0 < rank + ctot; p0 += 32) {
      const int32_t pp = p0 + lane;
      const bool valid = pp >= rank && pp < rank + ctot;
      uint32_t e = 0u;
      if (valid) {
        e = stage[pp - rank];
        gx[pp] = static_cast<int32_t>(e & 0x3FFFFFFFu);
      }
      const uint32_t ma = __ballot_sync(0xFFFFFFFFu, valid && ((e >> 30) & 1u));
      const uint32_t mb = __ballot_sync(0xFFFFFFFFu, valid && (e >> 31));
      if (lane == 0) {
        if (ma) atomicOr(&rka[p0 >> 5], ma);
        if (mb) atomicOr(&rkb[p0 >> 5], mb);
      }
    }
    __syncwarp();
    rank += ctot;
  }
  // padding of the last tile: any in-range key; its columns stay masked
  for (int64_t q = u + threadIdx.x; q < static_cast<int64_t>(ne) * bn; q += blockDim.x) gx[q] = 0;
  __syncthreads();
  const int wpt = bn >> 5;                       // mask words per tile
  for (int32_t c = threadIdx.x; c < ne; c += blockDim.x) {
    uint32_t ma[4] = {0u, 0u, 0u, 0u}, mb[4] = {0u, 0u, 0u, 0u};
    bool full = static_cast<int64_t>(c + 1) * bn <= u;
    for (int w = 0; w < wpt; ++w) {
      ma[w] = rka[c * wpt + w];
      mb[w] = rkb[c * wpt + w];
      full = full && ma[w] == 0xFFFFFFFFu;
      if (L.b_rows) full = full && mb[w] == 0xFFFFFFFFu;
    }
    uint4* d = reinterpret_cast<uint4*>(dw + c * 8);
    d[0] = make_uint4(ma[0], ma[1], ma[2], ma[3]);
    d[1] = make_uint4(mb[0], mb[1], mb[2], mb[3]);
    entries[e0 + c] = make_int2(static_cast<int32_t>((e0 + c) * bn),
                                full ? -1 : static_cast<int32_t>(e0 + c));
  }
}

// ---------------------------------------------------------------------------
// Key-major plans (64-row query tiles, TSR_ORIENT_KEYS): one work item per
// 64-query block with its own list, no union.  The list is cut into 64-key
// gathered tiles in list order; only the last tile can be partly filled (its
// unused slots are masked), every other tile is full.  gidx holds the lists
// back to back, each padded to whole tiles with key 0.

// One warp per 64-row query block: validate its list (indptr from 0 upward;
// keys ascending, unique, inside [0, N)) and count its tiles.  With slice_m =
// 128 the two 64-row halves of a block share its list.
__global__ void keylist_t_count_kernel(const int64_t* indptr, const int32_t* indices,
                                       int64_t n_items, int32_t nqb64, int32_t nqb, int32_t per,
                                       int32_t N, int32_t* cnt_e, int32_t* cnt_b,
                                       unsigned long long* tot, uint32_t* err) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= n_items) return;
  const int64_t bh = w / nqb64, qb = w % nqb64;
  const int64_t row = bh * nqb + qb / per;
  if (!list_ok(indptr, row)) {
    if (lane == 0) atomicOr(err, DEV_ERR_BAD_INPUT);
    return;
  }
  const int64_t b = indptr[row], e = indptr[row + 1];
  bool bad = false;
  for (int64_t base = b; base < e; base += 32) {
    const int64_t q = base + lane;
    const int32_t k = q < e ? indices[q] : INT32_MAX;
    int32_t nx = __shfl_down_sync(0xFFFFFFFFu, k, 1);
    if (lane == 31) nx = (q + 1 < e) ? indices[q + 1] : INT32_MAX;
    if (q < e && (k < 0 || k >= N || (q + 1 < e && nx <= k))) bad = true;
  }
  if (__any_sync(0xFFFFFFFFu, bad)) {
    if (lane == 0) atomicOr(err, DEV_ERR_BAD_INPUT);
    return;
  }
  if (lane == 0) {
    const int64_t len = e - b;
    const int32_t ne = static_cast<int32_t>((len + 63) / 64);
    const int32_t nb = (len % 64) ? 1 : 0;
    cnt_e[w] = ne;
    cnt_b[w] = nb;
    atomicAdd(&tot[0], static_cast<unsigned long long>(ne));
    atomicAdd(&tot[1], static_cast<unsigned long long>(nb));
    atomicMax(&tot[2], static_cast<unsigned long long>(ne));
  }
}

// One warp per 64-row query block: its list into gidx (tile t of the block at
// offset (ebegin + t) * 64, padding slots = key 0), the tiles' entries, and a
// list-form descriptor per tile (slot e for entry e) marking its listed slots.
__global__ void keylist_t_emit_kernel(const int64_t* indptr, const int32_t* indices,
                                      int64_t n_items, int32_t nqb64, int32_t nqb, int32_t per,
                                      const int32_t* cnt_e, const int32_t* ebegin, int2* entries,
                                      uint4* descs, int32_t* gidx) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= n_items) return;
  const int64_t bh = w / nqb64, qb = w % nqb64;
  const int64_t row = bh * nqb + qb / per;
  const int64_t b = indptr[row], len = indptr[row + 1] - b;
  const int64_t e0 = ebegin[w];
  const int32_t ne = cnt_e[w];
  int32_t* dst = gidx + e0 * 64;
  for (int64_t i = lane; i < static_cast<int64_t>(ne) * 64; i += 32) dst[i] = i < len ? indices[b + i] : 0;
  for (int32_t t = lane; t < ne; t += 32) {
    const int64_t valid = min(static_cast<int64_t>(64), len - static_cast<int64_t>(t) * 64);
    const uint32_t lo = valid >= 32 ? 0xFFFFFFFFu : ((1u << valid) - 1u);
    const uint32_t hi = valid >= 64 ? 0xFFFFFFFFu : (valid > 32 ? ((1u << (valid - 32)) - 1u) : 0u);
    const int64_t e = e0 + t;
    entries[e] = make_int2(static_cast<int32_t>(e * 64), valid == 64 ? -1 : static_cast<int32_t>(e));
    descs[2 * e] = make_uint4(lo, hi, 0u, 0u);
    descs[2 * e + 1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace

namespace {

// Key-major plan of a KEYLIST mask (the regime is known).
tsr_status plan_build_keylist_t(const tsr_mask* mask, const tsr_plan_opts* opts, const Regime& rg,
                                tsr_plan_impl* P, cudaStream_t stream) {
  const int32_t B = mask->B, H = mask->H, N = mask->N, M = mask->slice_m;
  const int32_t nqb64 = (N + 63) / 64, nqb = (N + M - 1) / M, per = M / 64;
  const int64_t n_items = static_cast<int64_t>(B) * H * nqb64;
  P->n_items = n_items;
  P->bn = 64;
  P->stages = rg.stages;
  P->ctas = rg.ctas;
  P->regime_id = rg.id;
  P->orient = TSR_ORIENT_KEYS;
  P->bm = 64;
  if (tsr_status s = devbuf_reserve(P->b_cnt, sizeof(int32_t) * 2 * n_items)) return s;
  int32_t* cnt_e = static_cast<int32_t*>(P->b_cnt.p);
  int32_t* cnt_b = cnt_e + n_items;
  unsigned long long* tot = static_cast<unsigned long long*>(P->b_tot.p);
  unsigned long long* host_tot = P->host_tot;
  const int threads = 256;
  const int64_t blocks_w = (n_items * 32 + threads - 1) / threads;
  if (n_items > 0) {
    keylist_t_count_kernel<<<static_cast<unsigned>(blocks_w), threads, 0, stream>>>(
        mask->indptr, mask->indices, n_items, nqb64, nqb, per, N, cnt_e, cnt_b, tot, P->err);
    TSR_CUDA(cudaGetLastError());
  }
  TSR_CUDA(cudaMemcpyAsync(host_tot + 8, P->err, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream));
  TSR_CUDA(cudaMemcpyAsync(host_tot, tot, sizeof(unsigned long long) * 3, cudaMemcpyDeviceToHost,
                           stream));
  TSR_CUDA(cudaStreamSynchronize(stream));
  if (static_cast<uint32_t>(host_tot[8] & 0xFFFFFFFFull) & DEV_ERR_BAD_INPUT)
    return fail(TSR_ERR_INVALID_ARG,
                "KEYLIST lists must be ascending, unique and inside [0, N), indptr from 0 upward");
  P->n_entries = static_cast<int64_t>(host_tot[0]);
  P->n_desc = P->n_entries;
  P->n_gidx = P->n_entries * 64;
  P->max_item_len = static_cast<int64_t>(host_tot[2]);
  if (P->n_gidx >= (int64_t{1} << 31))
    return fail(TSR_ERR_UNSUPPORTED, "gathered plan has more than 2^31 key slots");
  if (tsr_status s = devbuf_reserve(P->b_items, sizeof(tsr_plan_item) * n_items)) return s;
  if (tsr_status s = devbuf_reserve(P->b_entries, sizeof(tsr_plan_entry) * P->n_entries)) return s;
  if (tsr_status s = devbuf_reserve(P->b_descs, 32 * static_cast<size_t>(P->n_desc))) return s;
  if (tsr_status s = devbuf_reserve(P->b_gidx, sizeof(int32_t) * P->n_gidx)) return s;
  if (tsr_status s = devbuf_reserve(P->b_ebegin, sizeof(int32_t) * n_items)) return s;
  if (tsr_status s = devbuf_reserve(P->b_dbegin, sizeof(int32_t) * n_items)) return s;
  // a head's gathered key indices stream through L2 beside its K and V
  const int32_t group_heads =
      P->group_heads > 0 ? P->group_heads
                         : heads_per_group(N, P->d, static_cast<int64_t>(B) * H,
                                           4.0 * static_cast<double>(P->n_gidx) / (static_cast<double>(B) * H));
  const int64_t n_groups = (static_cast<int64_t>(B) * H + group_heads - 1) / group_heads;
  if (tsr_status s = devbuf_reserve(P->b_hist, sizeof(int32_t) * (n_groups * (P->max_item_len + 1) + 1)))
    return s;
  P->items = P->b_items.p;
  P->entries = P->b_entries.p;
  P->descs = P->b_descs.p;
  P->gidx = static_cast<int32_t*>(P->b_gidx.p);
  int32_t* ebegin = static_cast<int32_t*>(P->b_ebegin.p);
  const int lpt = (opts && (opts->flags & TSR_PLAN_NO_LPT)) ? 0 : 1;
  if (tsr_status s = plan_schedule_into(cnt_e, cnt_b, n_items, nqb64, H, lpt,
                                        static_cast<int32_t>(P->max_item_len), group_heads, ebegin,
                                        static_cast<int32_t*>(P->b_dbegin.p),
                                        static_cast<int32_t*>(P->b_hist.p), P->items, stream))
    return s;
  if (n_items > 0) {
    keylist_t_emit_kernel<<<static_cast<unsigned>(blocks_w), threads, 0, stream>>>(
        mask->indptr, mask->indices, n_items, nqb64, nqb, per, cnt_e, ebegin,
        static_cast<int2*>(P->entries), static_cast<uint4*>(P->descs), P->gidx);
    TSR_CUDA(cudaGetLastError());
  }
  return TSR_OK;
}

}  // namespace

tsr_status plan_build_keylist(const tsr_mask* mask, const tsr_plan_opts* opts, tsr_plan_impl* P,
                              cudaStream_t stream) {
  const int32_t B = mask->B, H = mask->H, N = mask->N, M = mask->slice_m;
  const int32_t nqt = (N + kBM - 1) / kBM, nqb = (N + M - 1) / M;
  const int64_t n_items = static_cast<int64_t>(B) * H * nqt;
  const int64_t n_lists = static_cast<int64_t>(B) * H * nqb;
  P->gathered = 1;
  P->slice_m = M;
  if (tsr_status s = devbuf_reserve(P->b_tot, sizeof(unsigned long long) * 8)) return s;
  if (!P->host_tot) TSR_CUDA(cudaMallocHost(&P->host_tot, sizeof(unsigned long long) * 9));
  unsigned long long* tot = static_cast<unsigned long long*>(P->b_tot.p);
  unsigned long long* host_tot = P->host_tot;
  TSR_CUDA(cudaMemsetAsync(tot, 0, sizeof(unsigned long long) * 8, stream));
  TSR_CUDA(cudaMemsetAsync(P->err, 0, sizeof(uint32_t), stream));
  const char* bad_lists =
      "KEYLIST lists must be ascending, unique and inside [0, N), indptr from 0 upward";
  // the lists' total length (density for the regime table, which picks the
  // tile orientation before the lists are counted)
  TSR_CUDA(cudaMemcpyAsync(host_tot + 6, mask->indptr, sizeof(int64_t), cudaMemcpyDeviceToHost, stream));
  TSR_CUDA(cudaMemcpyAsync(host_tot + 7, mask->indptr + n_lists, sizeof(int64_t),
                           cudaMemcpyDeviceToHost, stream));
  TSR_CUDA(cudaStreamSynchronize(stream));
  const int64_t first = static_cast<int64_t>(host_tot[6]), total = static_cast<int64_t>(host_tot[7]);
  if (first != 0 || total < 0) return fail(TSR_ERR_INVALID_ARG, bad_lists);
  if (!mask->indices && total > 0)
    return fail(TSR_ERR_INVALID_ARG, "indices is NULL but the key lists are not empty");
  P->n_logical_on = total;
  P->n_logical_total = n_lists * static_cast<int64_t>(N);
  const double density = static_cast<double>(total) / static_cast<double>(n_lists) / N;
  Regime rg;
  if (tsr_status s = resolve_regime(regime_lookup(TSR_MASK_KEYLIST, M, 1, N, density, P->d), opts,
                                    P->d, true, &rg))
    return s;
  if (rg.orient == TSR_ORIENT_KEYS) return plan_build_keylist_t(mask, opts, rg, P, stream);
  P->orient = TSR_ORIENT_ROWS;
  P->bm = kBM;
  P->n_items = n_items;
  if (tsr_status s = devbuf_reserve(P->b_cnt, sizeof(int32_t) * 3 * n_items)) return s;
  int32_t* cnt = static_cast<int32_t*>(P->b_cnt.p);
  const int threads = 256;
  const bool bitmap = N <= kBitmapMaxN;
  if (bitmap) {
    // validation runs inside the count kernel
    static bool attr_done[64] = {false};
    if (P->device < 0 || P->device >= 64 || !attr_done[P->device]) {
      TSR_CUDA(cudaFuncSetAttribute(keylist_count_bitmap_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(2 * 4 * bitmap_words16(kBitmapMaxN))));
      TSR_CUDA(cudaFuncSetAttribute(keylist_emit_bitmap_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(4 * emit_bitmap_words(kBitmapMaxN))));
      if (P->device >= 0 && P->device < 64) attr_done[P->device] = true;
    }
    if (n_items > 0) {
      keylist_count_bitmap_kernel<<<static_cast<unsigned>(n_items), 256,
                                    2 * 4 * static_cast<size_t>(bitmap_words16(N)), stream>>>(
          mask->indptr, mask->indices, n_items, nqt, nqb, M, N, cnt, tot, P->err);
      TSR_CUDA(cudaGetLastError());
    }
  } else {
    keylist_validate_kernel<<<static_cast<unsigned>((n_lists * 32 + threads - 1) / threads), threads,
                              0, stream>>>(mask->indptr, mask->indices, n_lists, N, P->err);
    TSR_CUDA(cudaGetLastError());
    TSR_CUDA(cudaMemcpyAsync(host_tot + 8, P->err, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream));
    TSR_CUDA(cudaStreamSynchronize(stream));
    if (static_cast<uint32_t>(host_tot[8] & 0xFFFFFFFFull) & DEV_ERR_BAD_INPUT)
      return fail(TSR_ERR_INVALID_ARG, bad_lists);
    keylist_count_kernel<<<static_cast<unsigned>((n_items * 32 + threads - 1) / threads), threads, 0,
                           stream>>>(mask->indptr, mask->indices, n_items, nqt, nqb, M, N, cnt, tot);
    TSR_CUDA(cudaGetLastError());
  }
  TSR_CUDA(cudaMemcpyAsync(host_tot + 8, P->err, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream));
  TSR_CUDA(cudaMemcpyAsync(host_tot, tot, sizeof(unsigned long long) * 8, cudaMemcpyDeviceToHost,
                           stream));
  TSR_CUDA(cudaStreamSynchronize(stream));
  if (static_cast<uint32_t>(host_tot[8] & 0xFFFFFFFFull) & DEV_ERR_BAD_INPUT)
    return fail(TSR_ERR_INVALID_ARG, bad_lists);

  P->bn = rg.bn;
  P->stages = rg.stages;
  P->ctas = rg.ctas;
  P->regime_id = rg.id;
  const int which = (rg.bn == 64) ? 0 : 1;
  P->n_entries = static_cast<int64_t>(host_tot[which]);
  P->n_desc = P->n_entries;
  P->n_gidx = P->n_entries * rg.bn;
  P->max_item_len = static_cast<int64_t>(host_tot[2 + which]);
  if (P->n_gidx >= (int64_t{1} << 31))
    return fail(TSR_ERR_UNSUPPORTED, "gathered plan has more than 2^31 key slots");

  if (tsr_status s = devbuf_reserve(P->b_items, sizeof(tsr_plan_item) * n_items)) return s;
  if (tsr_status s = devbuf_reserve(P->b_entries, sizeof(tsr_plan_entry) * P->n_entries)) return s;
  if (tsr_status s = devbuf_reserve(P->b_descs, 32 * static_cast<size_t>(P->n_desc))) return s;
  if (tsr_status s = devbuf_reserve(P->b_gidx, sizeof(int32_t) * P->n_gidx)) return s;
  if (tsr_status s = devbuf_reserve(P->b_ebegin, sizeof(int32_t) * n_items)) return s;
  if (tsr_status s = devbuf_reserve(P->b_dbegin, sizeof(int32_t) * n_items)) return s;
  // a head's gathered key indices stream through L2 beside its K and V
  const int32_t group_heads =
      P->group_heads > 0 ? P->group_heads
                         : heads_per_group(N, P->d, static_cast<int64_t>(B) * H,
                                           4.0 * static_cast<double>(P->n_gidx) / (static_cast<double>(B) * H));
  const int64_t n_groups = (static_cast<int64_t>(B) * H + group_heads - 1) / group_heads;
  if (tsr_status s = devbuf_reserve(P->b_hist, sizeof(int32_t) * (n_groups * (P->max_item_len + 1) + 1)))
    return s;
  P->items = P->b_items.p;
  P->entries = P->b_entries.p;
  P->descs = P->b_descs.p;
  P->gidx = static_cast<int32_t*>(P->b_gidx.p);
  int32_t* ebegin = static_cast<int32_t*>(P->b_ebegin.p);
  const int32_t* cnt_e = cnt + which * n_items;
  const int lpt = (opts && (opts->flags & TSR_PLAN_NO_LPT)) ? 0 : 1;
  if (tsr_status s = plan_schedule_into(cnt_e, cnt_e, n_items, nqt, H, lpt,
                                        static_cast<int32_t>(P->max_item_len), group_heads, ebegin,
                                        static_cast<int32_t*>(P->b_dbegin.p),
                                        static_cast<int32_t*>(P->b_hist.p), P->items, stream))
    return s;
  if (n_items > 0 && bitmap) {
    keylist_emit_bitmap_kernel<<<static_cast<unsigned>(n_items), 256, 4 * emit_bitmap_words(N),
                                 stream>>>(
        mask->indptr, mask->indices, nqt, nqb, M, N, rg.bn, cnt_e, ebegin,
        static_cast<int2*>(P->entries), static_cast<uint32_t*>(P->descs), P->gidx);
    TSR_CUDA(cudaGetLastError());
  } else if (n_items > 0) {
    keylist_emit_kernel<<<static_cast<unsigned>(n_items), 256, 0, stream>>>(
        mask->indptr, mask->indices, nqt, nqb, M, N, rg.bn, cnt_e, cnt + 2 * n_items, ebegin,
        static_cast<int2*>(P->entries), static_cast<uint32_t*>(P->descs), P->gidx);
    TSR_CUDA(cudaGetLastError());
  }
  return TSR_OK;
}

}  // namespace tsr
