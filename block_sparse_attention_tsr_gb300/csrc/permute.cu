// permute.cu -- temporal-major token permutation.
//
// Splash digest, "Splash Attention": token memory is permuted into temporal-
// major order so that the temporal pattern (same spatial index in every frame)
// reads contiguous rows.  With F frames of S tokens, token t = f*S + s moves to
// t' = s*F + f, so the F tokens that share spatial index s become one
// contiguous run and the temporal mask becomes block diagonal.
//
// The copy is HBM-bound: one 16-byte vector per thread, destination rows
// written in order (coalesced), source rows read whole (coalesced within a row).
#include <algorithm>

#include "internal.h"

namespace tsr {

namespace {

constexpr int kMaxPermHeads = 512;

struct PermParams {
  const uint4* src;
  uint4* dst;
  int64_t total;        // B * n_heads * N * vec
  int32_t B, H, N, F, S, vec, n_heads, inverse;
  int16_t heads[kMaxPermHeads];
};

__global__ void permute_rows_kernel(const __grid_constant__ PermParams p) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < p.total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t v = static_cast<int32_t>(i % p.vec);
    int64_t r = i / p.vec;
    const int32_t row = static_cast<int32_t>(r % p.N);
    r /= p.N;
    const int32_t hi = static_cast<int32_t>(r % p.n_heads);
    const int32_t b = static_cast<int32_t>(r / p.n_heads);
    const int64_t bh = static_cast<int64_t>(b) * p.H + p.heads[hi];
    int32_t src_row;
    if (!p.inverse) {
      src_row = (row % p.F) * p.S + row / p.F;   // dst row t' = s F + f  <-  t = f S + s
    } else {
      src_row = (row % p.S) * p.F + row / p.S;   // dst row t = f S + s  <-  t' = s F + f
    }
    p.dst[(bh * p.N + row) * p.vec + v] = p.src[(bh * p.N + src_row) * p.vec + v];
  }
}

}  // namespace

tsr_status launch_permute(const void* src, void* dst, int32_t B, int32_t H, int32_t F, int32_t S,
                          int32_t row_bytes, const int8_t* head_kind_host, int32_t inverse,
                          cudaStream_t stream) {
  PermParams p;
  p.src = static_cast<const uint4*>(src);
  p.dst = static_cast<uint4*>(dst);
  p.B = B;
  p.H = H;
  p.F = F;
  p.S = S;
  p.N = F * S;
  p.vec = row_bytes / 16;
  p.inverse = inverse;
  p.n_heads = 0;
  for (int32_t h = 0; h < H; ++h) {
    if (head_kind_host && head_kind_host[h] != TSR_HEAD_TEMPORAL) continue;
    if (p.n_heads == kMaxPermHeads) return fail(TSR_ERR_UNSUPPORTED, "more than 512 temporal heads");
    p.heads[p.n_heads++] = static_cast<int16_t>(h);
  }
  p.total = static_cast<int64_t>(B) * p.n_heads * p.N * p.vec;
  if (p.total == 0) return TSR_OK;
  const int threads = 256;
  int dev = 0;
  TSR_CUDA(cudaGetDevice(&dev));
  const int64_t blocks =
      std::min<int64_t>((p.total + threads - 1) / threads, static_cast<int64_t>(num_sms(dev)) * 8);
  permute_rows_kernel<<<static_cast<int>(blocks), threads, 0, stream>>>(p);
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

}  // namespace tsr
