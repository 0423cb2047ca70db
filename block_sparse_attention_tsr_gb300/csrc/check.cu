// check.cu -- device-side consistency checks of a tile plan (TSR_PLAN_DEBUG_CHECKS).
//
// The attention kernel trusts its plan: every work item's entry range, every key
// tile's coordinates, every boundary descriptor and every gathered key index are
// used as addresses.  These kernels read a finished plan and verify, without
// using any value as an address before it is checked:
//   * each item names a (b*h, query tile of the plan's height) inside the
//     problem, each pair exactly
//     once, with an entry range inside the plan and a layout of 0 or 1;
//   * contiguous entries: key tile starts inside [0, N), multiples of the tile
//     width, strictly ascending within an item; descriptor index -1 or inside
//     the plan; grid-form descriptors with 1..8 row and column segments,
//     ascending starts inside the tile; band-form descriptors with a frame
//     count of at least 1;
//   * gathered entries: tile e at gidx offset e * BN, descriptor index -1 or e,
//     and every gathered key index inside [0, N).
// A violation sets DEV_ERR_INTERNAL in the plan's error word; nothing traps.
#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace tsr {

namespace {

struct CheckArgs {
  const int4* items;
  const int2* entries;
  const uint8_t* descs;       // tsr_tile_desc, 32 bytes each
  const int32_t* gidx;
  int64_t n_items, n_entries, n_desc;
  int32_t BH, nqt, N, bm, bn, gathered;
  int32_t* seen;              // [BH * nqt], zeroed
  uint32_t* err;
};

__device__ __forceinline__ void flag(uint32_t* err) { atomicOr(err, DEV_ERR_INTERNAL); }

// One warp per work item.
__global__ void plan_check_items_kernel(CheckArgs a) {
  const int64_t it = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (it >= a.n_items) return;
  const int4 i0 = a.items[2 * it], i1 = a.items[2 * it + 1];
  const int32_t bh = i0.x, qt = i0.y, begin = i0.z, end = i0.w, layout = i1.x;
  if (bh < 0 || bh >= a.BH || qt < 0 || qt >= a.nqt || begin < 0 || end < begin ||
      end > a.n_entries || (layout != 0 && layout != 1)) {
    if (lane == 0) flag(a.err);
    return;
  }
  if (lane == 0) atomicAdd(&a.seen[static_cast<int64_t>(bh) * a.nqt + qt], 1);
  bool bad = false;
  for (int64_t e = begin + lane; e < end; e += 32) {
    const int2 en = a.entries[e];
    const int32_t kv = en.x, di = en.y;
    if (a.gathered) {
      bad |= static_cast<int64_t>(kv) != e * a.bn;
      bad |= !(di == -1 || (di == e && di < a.n_desc));
    } else {
      bad |= kv < 0 || kv >= a.N || kv % a.bn != 0;
      if (e > begin) bad |= a.entries[e - 1].x >= kv;
      bad |= !(di == -1 || (di >= 0 && di < a.n_desc));
      if (di >= 0 && di < a.n_desc) {
        const uint8_t* d = a.descs + static_cast<int64_t>(di) * 32;
        const int n_r = d[0], n_c = d[1];
        if (n_r == 0) {
          // band form: no segments, bits = F << 32 | R with F >= 1
          const uint32_t F = *reinterpret_cast<const uint32_t*>(d + 28);
          bad |= n_c != 0 || F < 1;
        } else {
          bad |= n_r > 8 || n_c < 1 || n_c > 8;
        }
        if (!(n_r < 1 || n_r > 8 || n_c < 1 || n_c > 8)) {
          bad |= d[2] != 0;                       // r_start[0]
          for (int r = 1; r < n_r; ++r) bad |= d[2 + r] <= d[1 + r] || d[2 + r] >= a.bm;
          bad |= d[10] != 0;                      // c_start[0]
          for (int c = 1; c <= n_c; ++c) bad |= d[10 + c] < d[9 + c];
          bad |= d[10 + n_c] > a.bn;
        }
      }
    }
  }
  if (a.gathered) {
    // every key slot of the item's tiles
    const int64_t s0 = static_cast<int64_t>(begin) * a.bn, s1 = static_cast<int64_t>(end) * a.bn;
    for (int64_t s = s0 + lane; s < s1; s += 32) bad |= a.gidx[s] < 0 || a.gidx[s] >= a.N;
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) flag(a.err);
}

// Every (b*h, query tile) must have exactly one item.
__global__ void plan_check_seen_kernel(const int32_t* seen, int64_t n, uint32_t* err) {
  bool bad = false;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    bad |= seen[i] != 1;
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) flag(err);
}

}  // namespace

tsr_status plan_check(const tsr_plan_impl* P, cudaStream_t stream) {
  const int32_t nqt = (P->N + P->bm - 1) / P->bm;
  const int64_t BH = static_cast<int64_t>(P->B) * P->H;
  const int64_t n_pairs = BH * nqt;
  void* seen = nullptr;
  TSR_CUDA(cudaMallocAsync(&seen, sizeof(int32_t) * static_cast<size_t>(n_pairs), stream));
  cudaError_t e = cudaMemsetAsync(seen, 0, sizeof(int32_t) * static_cast<size_t>(n_pairs), stream);
  if (e == cudaSuccess && P->n_items > 0) {
    CheckArgs a;
    a.items = static_cast<const int4*>(P->items);
    a.entries = static_cast<const int2*>(P->entries);
    a.descs = static_cast<const uint8_t*>(P->descs);
    a.gidx = P->gidx;
    a.n_items = P->n_items;
    a.n_entries = P->n_entries;
    a.n_desc = P->n_desc;
    a.BH = static_cast<int32_t>(BH);
    a.nqt = nqt;
    a.N = P->N;
    a.bm = P->bm;
    a.bn = P->bn;
    a.gathered = P->gathered;
    a.seen = static_cast<int32_t*>(seen);
    a.err = P->err;
    plan_check_items_kernel<<<static_cast<unsigned>((P->n_items * 32 + 255) / 256), 256, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
      plan_check_seen_kernel<<<static_cast<unsigned>(std::min<int64_t>(1024, (n_pairs + 255) / 256)),
                               256, 0, stream>>>(static_cast<const int32_t*>(seen), n_pairs, P->err);
      e = cudaGetLastError();
    }
  }
  const cudaError_t ef = cudaFreeAsync(seen, stream);
  if (e != cudaSuccess) return cuda_fail(e, "plan check");
  if (ef != cudaSuccess) return cuda_fail(ef, "plan check workspace");
  return TSR_OK;
}

}  // namespace tsr
