// route.cu -- SVG head routing by sampled queries.
//
// Sparse VideoGen digest, section "Sparse VideoGen": each attention head is
// assigned on the fly to a spatial or a temporal sparse pattern.  The pages give
// no criterion; the reading taken here: for sampled query rows, compare the
// head's attention output under each pattern with dense attention and send the
// head to the pattern with the smaller summed squared error.
//
// route_partial_kernel: one CTA of four warps per (b, h), 64 sampled rows (the
// host sorts the rows, so a CTA's rows span few frames) and one split of the
// keys (1,024 keys or more per split, so a 480p head gives 32 CTAs per row
// group).  Key chunks of 64 rows of K and V stream through a double-buffered
// shared-memory ring (cp.async).  Each warp computes S = Q K^T for its 16 rows
// with warp-level tensor-core MMAs (mma.sync m16n8k16, bf16 in, fp32 out) and
// runs two online softmaxes over the same scores: dense (every key) and spatial
// (the row's frame and frame 0; chunks no row of the warp reaches are skipped),
// each with its own P V accumulator, P taken straight from the score fragments.
// The split's (max, sum, unnormalised O) per row and pattern go to a workspace.
//
// route_combine_kernel: one warp per sampled row merges the splits of both
// patterns, computes the temporal pattern (F (2r + 1) keys per row) on CUDA
// cores with an online softmax, and adds |O_spatial - O_dense|^2,
// |O_temporal - O_dense|^2 and |O_dense|^2 into stats[b][h] (fp32 atomics).
// route_finish_kernel sums over b and writes head_kind[h] = temporal iff its
// error is smaller.
//
// Work: about 4 * n_samples * N * d flops per head for the dense pattern (0.5
// GFLOP per head at 64 samples and 480p) plus up to a third more for the
// spatial one.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <string>

#include "internal.h"

namespace tsr {

namespace {

constexpr int kRouteRows = 64;        // sampled rows per CTA (16 per warp)
constexpr int kRouteKeys = 64;        // keys per staged chunk
constexpr int kRouteMaxSamples = 1024;

struct RouteParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  float* stats;                // [B*H][3]
  float* ws;                   // [B*H][row groups][splits][2][64][2 + D]
  int32_t N, F, S, R, n_samples;
  int32_t n_splits, keys_per_split;
  float scale_log2;            // log2(e) / sqrt(d)
  int32_t samples[kRouteMaxSamples];   // ascending
};

__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, bool valid) {
  // 16-byte async copy; with valid == false nothing is read and zeros are written
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16) * B (16x8 bf16)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Online-softmax state of one pattern for the thread's two rows (g, g + 8):
// running maxima, partial row sums, and the P V accumulator fragments.
template <int D>
struct PatternAcc {
  float m[2], l[2];
  float o[D / 8][4];
  __device__ void init() {
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  }
  // x: scores (log2 units) of the chunk, allowed by bits ok[nt] (bit c: row g,
  // key 2t + (c & 1); bits 2, 3: row g + 8); v_base: the chunk's V rows.
  __device__ void update(const float (&x)[kRouteKeys / 8][4], const uint32_t (&ok)[kRouteKeys / 8],
                         uint32_t v_base, int lane) {
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < kRouteKeys / 8; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if ((ok[nt] >> c) & 1u) mx[c >> 1] = fmaxf(mx[c >> 1], x[nt][c]);
    float alpha[2], mu[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xFFFFFFFFu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xFFFFFFFFu, mx[h], 2));
      const float m_new = fmaxf(m[h], mx[h]);
      // a row with no allowed key so far keeps O = 0 and l = 0
      alpha[h] = (m_new == -INFINITY) ? 1.f : exp2f(m[h] - m_new);
      mu[h] = (m_new == -INFINITY) ? 0.f : m_new;
      m[h] = m_new;
    }
    uint32_t pa[kRouteKeys / 16][4];
    float ls[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < kRouteKeys / 8; ++nt) {
      float p[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        p[c] = ((ok[nt] >> c) & 1u) ? exp2f(x[nt][c] - mu[c >> 1]) : 0.f;
        ls[c >> 1] += p[c];
      }
      // score fragment (16x8) -> half of an A fragment (16x16) of P
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack2(p[0], p[1]);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack2(p[2], p[3]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) l[h] = l[h] * alpha[h] + ls[h];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
    // O += P V: V rows (keys) are the K dimension; ldmatrix .trans yields the
    // B fragments of two 8-column output tiles at a time
#pragma unroll
    for (int ks = 0; ks < kRouteKeys / 16; ++ks) {
      const uint32_t a[4] = {pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3]};
#pragma unroll
      for (int n = 0; n < D / 8; n += 2) {
        uint32_t b[4];
        const int key = ks * 16 + (lane & 15);
        const int col = n * 8 + (lane >> 4) * 8;
        ldsm_x4_t(v_base + (key * (D + 8) + col) * 2, b);
        mma16816(o[n], a, b[0], b[1]);
        mma16816(o[n + 1], a, b[2], b[3]);
      }
    }
  }
};

template <int D>
__global__ void __launch_bounds__(128) route_partial_kernel(const __grid_constant__ RouteParams p) {
  constexpr int LD = D + 8;                         // padded row (bf16 elements)
  constexpr int TILE = kRouteRows * LD;             // elements of one staged tile
  constexpr int REC = 2 + D;                        // per row and pattern: m, l, O[D]
  extern __shared__ __align__(16) __nv_bfloat16 smem[];
  __nv_bfloat16* sQ = smem;
  __nv_bfloat16* sK = smem + TILE;                  // [2][kRouteKeys][LD]
  __nv_bfloat16* sV = smem + 3 * TILE;              // [2][kRouteKeys][LD]
  __shared__ int32_t rows_i[kRouteRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t bh = blockIdx.x;
  const int rg = blockIdx.y, split = blockIdx.z;
  const size_t head = static_cast<size_t>(bh) * p.N * D;
  const int row0 = rg * kRouteRows;
  if (threadIdx.x < kRouteRows) {
    const int sidx = row0 + threadIdx.x;
    // rows past the sample count repeat the last sample (keeps the rows sorted);
    // the combine step leaves them out
    rows_i[threadIdx.x] = p.samples[sidx < p.n_samples ? sidx : p.n_samples - 1];
  }
  __syncthreads();
  constexpr int UPR = D / 8;                        // 16-byte units per row
  for (int u = threadIdx.x; u < kRouteRows * UPR; u += blockDim.x) {
    const int r = u / UPR, c = u % UPR;
    cp16(su32(sQ + r * LD + c * 8), p.q + head + static_cast<size_t>(rows_i[r]) * D + c * 8, true);
  }
  const int k_begin = split * p.keys_per_split;
  const int k_end = min(p.N, k_begin + p.keys_per_split);
  auto stage = [&](int chunk, int buf) {
    const int j0 = k_begin + chunk * kRouteKeys;
    for (int u = threadIdx.x; u < kRouteKeys * UPR; u += blockDim.x) {
      const int r = u / UPR, c = u % UPR;
      const bool in = j0 + r < k_end;
      const size_t off = head + static_cast<size_t>(in ? j0 + r : 0) * D + c * 8;
      cp16(su32(sK + (buf * kRouteKeys + r) * LD + c * 8), p.k + off, in);
      cp16(su32(sV + (buf * kRouteKeys + r) * LD + c * 8), p.v + off, in);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  const int n_chunks = (k_end - k_begin + kRouteKeys - 1) / kRouteKeys;
  stage(0, 0);
  const int r0 = warp * 16 + g, r1 = r0 + 8;
  const int fr0 = rows_i[r0] / p.S, fr1 = rows_i[r1] / p.S;
  const int wf_lo = rows_i[warp * 16] / p.S, wf_hi = rows_i[warp * 16 + 15] / p.S;
  PatternAcc<D> dense, spat;
  dense.init();
  spat.init();
  for (int chunk = 0; chunk < n_chunks; ++chunk) {
    const int buf = chunk & 1;
    if (chunk + 1 < n_chunks) {
      stage(chunk + 1, buf ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const int j0 = k_begin + chunk * kRouteKeys;
    const __nv_bfloat16* kb = sK + buf * kRouteKeys * LD;
    float x[kRouteKeys / 8][4];
#pragma unroll
    for (int nt = 0; nt < kRouteKeys / 8; ++nt) x[nt][0] = x[nt][1] = x[nt][2] = x[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(su32(sQ + (warp * 16 + (lane & 15)) * LD + ks * 16 + (lane >> 4) * 8), a);
#pragma unroll
      for (int nt = 0; nt < kRouteKeys / 8; nt += 2) {
        uint32_t b[4];
        // matrices: keys nt*8.., dims ks*16 | +8, keys (nt+1)*8.., dims ks*16 | +8
        const int key = nt * 8 + (lane & 7) + ((lane >> 4) << 3);
        const int col = ks * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4(su32(kb + key * LD + col), b);
        mma16816(x[nt], a, b[0], b[1]);
        mma16816(x[nt + 1], a, b[2], b[3]);
      }
    }
    uint32_t ok_d[kRouteKeys / 8], ok_s[kRouteKeys / 8];
#pragma unroll
    for (int nt = 0; nt < kRouteKeys / 8; ++nt) {
      ok_d[nt] = ok_s[nt] = 0u;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = j0 + nt * 8 + 2 * t + (c & 1);
        const int fr = (c >> 1) ? fr1 : fr0;
        x[nt][c] *= p.scale_log2;
        if (j < k_end) {
          ok_d[nt] |= 1u << c;
          if (j < p.S || j / p.S == fr) ok_s[nt] |= 1u << c;
        }
      }
    }
    const uint32_t vb = su32(sV + buf * kRouteKeys * LD);
    dense.update(x, ok_d, vb, lane);
    // the spatial pattern reaches this chunk only through frame 0 or the
    // frames of the warp's rows
    const bool reach = j0 < p.S || (j0 + kRouteKeys > wf_lo * p.S && j0 < (wf_hi + 1) * p.S);
    if (reach) spat.update(x, ok_s, vb, lane);
    __syncthreads();
  }
  // this split's (max, full row sum, unnormalised O) per row and pattern
  float* w = p.ws + ((bh * gridDim.y + rg) * p.n_splits + split) * (2 * kRouteRows * REC);
#pragma unroll
  for (int pat = 0; pat < 2; ++pat) {
    const PatternAcc<D>& acc = pat ? spat : dense;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float l = acc.l[h];
      l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
      l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);
      float* rec = w + (pat * kRouteRows + (h ? r1 : r0)) * REC;
      if (t == 0) {
        rec[0] = acc.m[h];
        rec[1] = l;
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
        *reinterpret_cast<float2*>(rec + 2 + n * 8 + 2 * t) =
            make_float2(acc.o[n][2 * h], acc.o[n][2 * h + 1]);
    }
  }
}

// One warp per sampled row: merge the splits, then the temporal pattern and
// the error sums.
template <int D>
__global__ void __launch_bounds__(256) route_combine_kernel(const __grid_constant__ RouteParams p,
                                                            int32_t n_row_groups, int64_t n_heads) {
  constexpr int REC = 2 + D;
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t bh = wid / (static_cast<int64_t>(n_row_groups) * kRouteRows);
  const int rs = static_cast<int>(wid % (static_cast<int64_t>(n_row_groups) * kRouteRows));
  if (bh >= n_heads) return;
  if (rs >= p.n_samples) return;
  const int rg = rs / kRouteRows, row = rs % kRouteRows;
  const int i = p.samples[rs];
  const size_t head = static_cast<size_t>(bh) * p.N * D;
  const float* w0 = p.ws + (bh * n_row_groups + rg) * static_cast<int64_t>(p.n_splits) * (2 * kRouteRows * REC);
  float o[2][E];
#pragma unroll
  for (int pat = 0; pat < 2; ++pat) {
    float M = -INFINITY;
    for (int sp = 0; sp < p.n_splits; ++sp)
      M = fmaxf(M, w0[(sp * 2 + pat) * kRouteRows * REC + row * REC]);
    float L = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[pat][e] = 0.f;
    for (int sp = 0; sp < p.n_splits; ++sp) {
      const float* rec = w0 + ((sp * 2 + pat) * kRouteRows + row) * REC;
      const float m = rec[0];
      if (m == -INFINITY) continue;
      const float f = exp2f(m - M);
      L = fmaf(rec[1], f, L);
#pragma unroll
      for (int e = 0; e < E; ++e) o[pat][e] = fmaf(rec[2 + lane * E + e], f, o[pat][e]);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) o[pat][e] /= L;
  }
  // temporal pattern: keys f*S + s' with |s' - s_i| <= R, online softmax
  const int s_i = i % p.S;
  const int lo = max(0, s_i - p.R), hi = min(p.S - 1, s_i + p.R), wl = hi - lo + 1;
  float qv[E];
#pragma unroll
  for (int e = 0; e < E; ++e)
    qv[e] = __bfloat162float(p.q[head + static_cast<size_t>(i) * D + lane * E + e]) * p.scale_log2;
  float m = -INFINITY, l = 0.f, ot[E];
#pragma unroll
  for (int e = 0; e < E; ++e) ot[e] = 0.f;
  for (int kk = 0; kk < p.F * wl; ++kk) {
    const size_t j = static_cast<size_t>(kk / wl) * p.S + lo + kk % wl;
    float s = 0.f, vv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      s = fmaf(qv[e], __bfloat162float(p.k[head + j * D + lane * E + e]), s);
      vv[e] = __bfloat162float(p.v[head + j * D + lane * E + e]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
    const float m_new = fmaxf(m, s);
    const float a = exp2f(m - m_new), pk = exp2f(s - m_new);
    l = l * a + pk;
#pragma unroll
    for (int e = 0; e < E; ++e) ot[e] = fmaf(pk, vv[e], ot[e] * a);
    m = m_new;
  }
  float err_s = 0.f, err_t = 0.f, den = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float od = o[0][e], ds = o[1][e] - od, dt = ot[e] / l - od;
    err_s = fmaf(ds, ds, err_s);
    err_t = fmaf(dt, dt, err_t);
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
  // the sums do not depend on the order of the rows; sorted rows keep a CTA's
  // rows in few frames
  std::copy(samples, samples + n_samples, prm.samples);
  std::sort(prm.samples, prm.samples + n_samples);
  for (int s = n_samples; s < kRouteMaxSamples; ++s) prm.samples[s] = 0;
  const int64_t n_heads = static_cast<int64_t>(B) * H;
  const int32_t n_rg = (n_samples + kRouteRows - 1) / kRouteRows;
  // keys per split: at least 1,024, more when the workspace would pass 256 MB
  const size_t rec_bytes = static_cast<size_t>(2) * kRouteRows * (2 + d) * 4;
  int64_t kps = 1024;
  while (static_cast<size_t>(n_heads) * n_rg * ((prm.N + kps - 1) / kps) * rec_bytes >
         (static_cast<size_t>(256) << 20))
    kps *= 2;
  prm.keys_per_split = static_cast<int32_t>(std::min<int64_t>(kps, prm.N));
  prm.n_splits = (prm.N + prm.keys_per_split - 1) / prm.keys_per_split;
  const size_t ws_bytes = static_cast<size_t>(n_heads) * n_rg * prm.n_splits * rec_bytes;
  void* ws = nullptr;
  TSR_CUDA(cudaMallocAsync(&ws, ws_bytes, stream));
  prm.ws = static_cast<float*>(ws);
  TSR_CUDA(cudaMemsetAsync(stats, 0, sizeof(float) * 3 * static_cast<size_t>(n_heads), stream));
  const dim3 grid(static_cast<unsigned>(n_heads), static_cast<unsigned>(n_rg),
                  static_cast<unsigned>(prm.n_splits));
  const size_t smem = static_cast<size_t>(5) * kRouteRows * (d + 8) * 2;
  const int64_t warps = n_heads * n_rg * kRouteRows;
  const unsigned cblocks = static_cast<unsigned>((warps + 7) / 8);
  cudaError_t e;
  if (d == 128) {
    e = cudaFuncSetAttribute(route_partial_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) {
      route_partial_kernel<128><<<grid, 128, smem, stream>>>(prm);
      route_combine_kernel<128><<<cblocks, 256, 0, stream>>>(prm, n_rg, n_heads);
    }
  } else {
    e = cudaFuncSetAttribute(route_partial_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess) {
      route_partial_kernel<64><<<grid, 128, smem, stream>>>(prm);
      route_combine_kernel<64><<<cblocks, 256, 0, stream>>>(prm, n_rg, n_heads);
    }
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  const cudaError_t ef = cudaFreeAsync(ws, stream);
  if (e != cudaSuccess) return fail(TSR_ERR_CUDA, std::string("route kernels: ") + cudaGetErrorString(e));
  if (ef != cudaSuccess) return fail(TSR_ERR_CUDA, std::string("cudaFreeAsync: ") + cudaGetErrorString(ef));
  route_finish_kernel<<<1, 256, 0, stream>>>(stats, B, H, head_kind);
  TSR_CUDA(cudaGetLastError());
  return TSR_OK;
}

}  // namespace tsr
