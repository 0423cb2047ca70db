// route.cu -- SVG head routing by sampled queries.
//
// Sparse VideoGen digest, section "Sparse VideoGen": each attention head is
// assigned on the fly to a spatial or a temporal sparse pattern.  The pages give
// no criterion; the reading taken here: for sampled query rows, compare the
// head's attention output under each pattern with dense attention and send the
// head to the pattern with the smaller summed squared error.
//
// route_kernel: one warp per sampled query row of one (b, h).  The block's
// eight warps share 32-key chunks of K and V staged in shared memory; lane l
// scores key j0 + l, and three online softmaxes run side by side over the same
// scores -- dense (every key), spatial (the query's frame and frame 0) and
// temporal (spatial index within the radius) -- each with its own running
// maximum, sum and output (lane l holds output dimensions l, l + 32, ...).
// Chunks where a pattern allows no key are skipped for it.  At the end each
// warp adds |O_spatial - O_dense|^2, |O_temporal - O_dense|^2 and |O_dense|^2
// into stats[b][h] (fp32 atomics).  route_finish_kernel sums over b and writes
// head_kind[h] = temporal iff its error is smaller.
//
// The arithmetic is fp32 on CUDA cores: the step costs about 4 * n_samples * N * d
// flops per head (0.5 GFLOP per head at 64 samples and 480p), far below one
// attention call, and it is not a tensor-shaped contraction per warp.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace tsr {

namespace {

constexpr int kRouteWarps = 8;        // sampled rows per block
constexpr int kRouteChunk = 32;       // keys per staged chunk
constexpr int kRouteMaxSamples = 1024;

struct RouteParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  float* stats;                // [B*H][3]
  int32_t N, F, S, R, n_samples;
  float scale_log2;            // log2(e) / sqrt(d)
  int32_t samples[kRouteMaxSamples];
};

template <int D>
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(const __grid_constant__ RouteParams p) {
  constexpr int E = D / 32;                 // output dimensions per lane
  constexpr int W2 = D / 2;                 // bf16 pairs per row
  __shared__ __align__(16) __nv_bfloat162 sk[kRouteChunk][W2];
  __shared__ __align__(16) __nv_bfloat16 sv[kRouteChunk][D];
  __shared__ float2 sq[kRouteWarps][W2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bh = blockIdx.x;
  const int si_idx = blockIdx.y * kRouteWarps + warp;
  const bool active = si_idx < p.n_samples;
  const int32_t i = active ? p.samples[si_idx] : 0;
  const size_t head = static_cast<size_t>(bh) * p.N * D;
  // the query row, scaled into the log2 domain
  for (int w = lane; w < W2; w += 32) {
    const __nv_bfloat162 x = reinterpret_cast<const __nv_bfloat162*>(p.q + head + static_cast<size_t>(i) * D)[w];
    sq[warp][w] = make_float2(__bfloat162float(x.x) * p.scale_log2, __bfloat162float(x.y) * p.scale_log2);
  }
  const int fi = i / p.S, s_i = i % p.S;
  float m[3], l[3], o[3][E];
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    m[t] = -INFINITY;
    l[t] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[t][e] = 0.f;
  }
  for (int32_t j0 = 0; j0 < p.N; j0 += kRouteChunk) {
    __syncthreads();
    // stage K and V rows j0 .. j0 + 31 (16-byte units; rows past N read as 0)
    constexpr int UNITS = kRouteChunk * D * 2 / 16;
    for (int u = threadIdx.x; u < UNITS; u += blockDim.x) {
      const int row = u / (D * 2 / 16), col = u % (D * 2 / 16);
      uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
      if (j0 + row < p.N) {
        const size_t off = head + static_cast<size_t>(j0 + row) * D;
        kx = reinterpret_cast<const uint4*>(p.k + off)[col];
        vx = reinterpret_cast<const uint4*>(p.v + off)[col];
      }
      reinterpret_cast<uint4*>(&sk[row][0])[col] = kx;
      reinterpret_cast<uint4*>(&sv[row][0])[col] = vx;
    }
    __syncthreads();
    if (!active) continue;
    // lane's key: j = j0 + lane; pairs visited in a lane-rotated order so the
    // 32 lanes read 32 different banks
    const int32_t j = j0 + lane;
    float s = 0.f;
#pragma unroll 8
    for (int c = 0; c < W2; ++c) {
      const int w = (c + lane) % W2;
      const float2 kf = __bfloat1622float2(sk[lane][w]);
      const float2 qf = sq[warp][w];
      s = fmaf(qf.x, kf.x, s);
      s = fmaf(qf.y, kf.y, s);
    }
    const bool in_range = j < p.N;
    const int sj = j % p.S;
    const bool allow[3] = {in_range, in_range && (j / p.S == fi || j < p.S),
                           in_range && abs(sj - s_i) <= p.R};
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      if (!__any_sync(0xFFFFFFFFu, allow[t])) continue;
      float cm = allow[t] ? s : -INFINITY;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, off));
      const float m_new = fmaxf(m[t], cm);
      const float alpha = exp2f(m[t] - m_new);      // 0 while m[t] is -inf
      const float pj = allow[t] ? exp2f(s - m_new) : 0.f;
      float ps = pj;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, off);
      l[t] = l[t] * alpha + ps;
      m[t] = m_new;
#pragma unroll
      for (int e = 0; e < E; ++e) o[t][e] *= alpha;
      for (int r = 0; r < kRouteChunk; ++r) {
        const float pr = __shfl_sync(0xFFFFFFFFu, pj, r);
        if (pr == 0.f) continue;                      // warp-uniform
#pragma unroll
        for (int e = 0; e < E; ++e) o[t][e] = fmaf(pr, __bfloat162float(sv[r][lane + 32 * e]), o[t][e]);
      }
    }
  }
  if (!active) return;
  float err_s = 0.f, err_t = 0.f, den = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float od = o[0][e] / l[0], os = o[1][e] / l[1], ot = o[2][e] / l[2];
    err_s = fmaf(os - od, os - od, err_s);
    err_t = fmaf(ot - od, ot - od, err_t);
    den = fmaf(od, od, den);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    err_s += __shfl_xor_sync(0xFFFFFFFFu, err_s, off);
    err_t += __shfl_xor_sync(0xFFFFFFFFu, err_t, off);
    den += __shfl_xor_sync(0xFFFFFFFFu, den, off);
  }
  if (lane == 0) {
    atomicAdd(&p.stats[3 * bh + 0], err_s);
    atomicAdd(&p.stats[3 * bh + 1], err_t);
    atomicAdd(&p.stats[3 * bh + 2], den);
  }
}

__global__ void route_finish_kernel(const float* stats, int32_t B, int32_t H, int8_t* head_kind) {
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    double es = 0.0, et = 0.0;
    for (int b = 0; b < B; ++b) {
      es += stats[3 * (static_cast<int64_t>(b) * H + h) + 0];
      et += stats[3 * (static_cast<int64_t>(b) * H + h) + 1];
    }
    head_kind[h] = et < es ? static_cast<int8_t>(TSR_HEAD_TEMPORAL) : static_cast<int8_t>(TSR_HEAD_SPATIAL);
  }
}

}  // namespace

tsr_status launch_route(const void* q, const void* k, const void* v, int32_t B, int32_t H,
                        int32_t F, int32_t S, int32_t d, int32_t R, const int32_t* samples,
                        int32_t n_samples, float* stats, int8_t* head_kind, cudaStream_t stream) {
  if (n_samples > kRouteMaxSamples)
    return fail(TSR_ERR_UNSUPPORTED, "at most 1024 sampled rows per call");
  RouteParams prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k = static_cast<const __nv_bfloat16*>(k);
  prm.v = static_cast<const __nv_bfloat16*>(v);
  prm.stats = stats;
  prm.N = F * S;
  prm.F = F;
  prm.S = S;
  prm.R = R;
  prm.n_samples = n_samples;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  for (int s = 0; s < kRouteMaxSamples; ++s) prm.samples[s] = s < n_samples ? samples[s] : 0;
  TSR_CUDA(cudaMemsetAsync(stats, 0, sizeof(float) * 3 * static_cast<size_t>(B) * H, stream));
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(B) * H),
                  static_cast<unsigned>((n_samples + kRouteWarps - 1) / kRouteWarps));
  if (d == 128)
    route_kernel<128><<<grid, kRouteWarps * 32, 0, stream>>>(prm);
  else
    route_kernel<64><<<grid, kRouteWarps * 32, 0, stream>>>(prm);
  TSR_CUDA(cudaGetLastError());
  route_finish_kernel<<<1, 256, 0, stream>>>(stats, B, H, head_kind);
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

}  // namespace tsr
