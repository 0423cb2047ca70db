// svg_temporal.cu -- the temporal heads of an SVG mask, by spatial position.
//
// Sparse VideoGen digest, "Sparse VideoGen": a temporal head lets a token see
// the tokens at the same spatial position in every frame.  With radius 0 the
// token t = f S + s (frame f, spatial index s) sees exactly the F keys
// f' S + s, f' = 0 .. F-1, so a temporal head is S independent F x F attention
// blocks, one per spatial position.  On the attention tiles such a head wastes
// most of each tile (a 128-row temporal-major tile holds six 21 x 21 blocks on
// its diagonal) and gathers every row through the permutation; here the work
// is bound by HBM: each block reads its F rows of Q, K and V once and writes F
// rows of O (4 F d 2 bytes per position, plus 4 F of lse).
//
// One warp per (head, spatial position), four per CTA, no CTA-wide barrier:
//   - the warp copies the block's F rows of Q, K and V into its shared memory
//     with 16-byte cp.async (rows of d bf16, 16-byte units swizzled by row so
//     that eight rows at one column fall in eight different bank groups);
//   - S = Q K^T on the tensor cores as warp-level m16n8k16 bf16 MMAs with fp32
//     accumulators, the block padded to 16 or 32 query rows and to 8-key tiles
//     (padding rows read row F - 1, padding keys get -inf);
//   - softmax in registers (row maximum and sum across the four lanes that
//     hold a row), P rounded to bf16 as the next MMA's A operand;
//   - O = P V (V through ldmatrix.trans), divided by the row sum, staged as
//     bf16 in the shared memory Q held and stored as whole 16-byte units;
//   - lse = ln 2 (m + log2 l).  Every row has its own key, so none is empty.
// The blocks are at most 32 x 32: a warp-level MMA covers one with no more
// padding than the 16 x 8 fragment shape, where the 64- or 128-row tensor-core
// tiles would be mostly padding.  CTAs of spatial heads return at once.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace tsr {

namespace {

constexpr int kWarps = 4;        // spatial positions per CTA
constexpr int kMaxF = 32;        // frames per position handled here

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// D += A B, m16n8k16: A row-major bf16, B column-major bf16, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte unit c of row r in a swizzled [rows][D] bf16 array.
template <int D>
__device__ __forceinline__ uint32_t sw(int r, int c) {
  return static_cast<uint32_t>(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32) svg_temporal_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
    const int8_t* __restrict__ head_kind, int32_t H, int32_t N, int32_t F, int32_t S, int64_t bh_lo,
    float scale_log2) {
  constexpr int U = D / 8;                                   // 16-byte units per row
  constexpr int NT = D / 8;                                  // 8-column tiles of O
  extern __shared__ __align__(128) uint8_t dyn[];
  const int64_t bh = bh_lo + blockIdx.y;
  if (head_kind[bh % H] != TSR_HEAD_TEMPORAL) return;        // uniform over the CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t s = blockIdx.x * kWarps + warp;
  if (s >= S) return;                                        // no CTA-wide sync below
  const size_t head = static_cast<size_t>(bh) * N * D;
  const uint32_t tensor_bytes = static_cast<uint32_t>(F * D * 2);
  const uint32_t qs = smem_u32(dyn) + warp * 3 * tensor_bytes;
  const uint32_t ks = qs + tensor_bytes;
  const uint32_t vs = ks + tensor_bytes;

  // 1. rows f S + s of Q, K and V -> shared memory
  {
    const __nv_bfloat16* src[3] = {q + head, k + head, v + head};
    const uint32_t dst[3] = {qs, ks, vs};
#pragma unroll
    for (int t = 0; t < 3; ++t)
      for (int u = lane; u < F * U; u += 32) {
        const int f = u / U, c = u % U;
        cp_async_16(dst[t] + sw<D>(f, c), src[t] + (static_cast<size_t>(f) * S + s) * D + c * 8);
      }
    cp_async_commit();
    cp_async_wait_all();
    __syncwarp();
  }

  const int g = lane >> 2, tq = lane & 3;                    // fragment row, column pair
  const int n_m = (F + 15) >> 4;                             // 16-row query tiles: 1 or 2
  const int n_n = (F + 7) >> 3;                              // 8-key tiles: 1 .. 4
  const int n_k = (F + 15) >> 4;                             // 16-key steps of P V: 1 or 2
  for (int mt = 0; mt < n_m; ++mt) {
    // 2. S = Q K^T for query rows [16 mt, 16 mt + 16) and keys [0, 8 n_n)
    float sacc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
    const int arow = min(mt * 16 + (lane & 15), F - 1);
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2) {
      uint32_t a[2][4];
      ldsm_x4(qs + sw<D>(arow, 2 * kk + (lane >> 4)), a[0][0], a[0][1], a[0][2], a[0][3]);
      ldsm_x4(qs + sw<D>(arow, 2 * kk + 2 + (lane >> 4)), a[1][0], a[1][1], a[1][2], a[1][3]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        if (nt < n_n) {
          const int brow = min(nt * 8 + (lane & 7), F - 1);
          uint32_t b0, b1, b2, b3;                           // key tile nt, units 2kk .. 2kk + 3
          ldsm_x4(ks + sw<D>(brow, 2 * kk + (lane >> 3)), b0, b1, b2, b3);
          mma_bf16(sacc[nt], a[0][0], a[0][1], a[0][2], a[0][3], b0, b1);
          mma_bf16(sacc[nt], a[1][0], a[1][1], a[1][2], a[1][3], b2, b3);
        }
      }
    }
    // 3. softmax of rows g and g + 8 of the tile (keys past F are -inf)
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool ok = nt < n_n && nt * 8 + 2 * tq + e < F;
        sacc[nt][e] = ok ? sacc[nt][e] * scale_log2 : -INFINITY;
        sacc[nt][2 + e] = ok ? sacc[nt][2 + e] * scale_log2 : -INFINITY;
        m0 = fmaxf(m0, sacc[nt][e]);
        m1 = fmaxf(m1, sacc[nt][2 + e]);
      }
    }
    m0 = fmaxf(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, 1));
    m0 = fmaxf(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, 2));
    m1 = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, 1));
    m1 = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, 2));
    float l0 = 0.f, l1 = 0.f;
    uint32_t p[4][2];                                        // bf16 pairs of rows g, g + 8
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float e0 = ex2_approx(sacc[nt][0] - m0), e1 = ex2_approx(sacc[nt][1] - m0);
      const float e2 = ex2_approx(sacc[nt][2] - m1), e3 = ex2_approx(sacc[nt][3] - m1);
      l0 += e0 + e1;
      l1 += e2 + e3;
      p[nt][0] = pack_bf16x2(e0, e1);
      p[nt][1] = pack_bf16x2(e2, e3);
    }
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
    l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
    l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
    // 4. O = P V over keys [0, 16 n_k)
    float oacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) oacc[nt][0] = oacc[nt][1] = oacc[nt][2] = oacc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      if (kk < n_k) {
        const int vrow = min(kk * 16 + (lane & 15), F - 1);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          uint32_t b0, b1, b2, b3;                           // column tiles 2np and 2np + 1
          ldsm_x4_trans(vs + sw<D>(vrow, 2 * np + (lane >> 4)), b0, b1, b2, b3);
          mma_bf16(oacc[2 * np], p[2 * kk][0], p[2 * kk][1], p[2 * kk + 1][0], p[2 * kk + 1][1],
                   b0, b1);
          mma_bf16(oacc[2 * np + 1], p[2 * kk][0], p[2 * kk][1], p[2 * kk + 1][0],
                   p[2 * kk + 1][1], b2, b3);
        }
      }
    }
    // 5. O / l as bf16 into this tile's rows of the Q buffer (which only this
    // tile read), and lse
    __syncwarp();
    const float i0 = 1.f / l0, i1 = 1.f / l1;
    const int r0 = mt * 16 + g, r1 = r0 + 8;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (r0 < F)
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(qs + sw<D>(r0, nt) + 4 * tq),
                     "r"(pack_bf16x2(oacc[nt][0] * i0, oacc[nt][1] * i0))
                     : "memory");
      if (r1 < F)
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(qs + sw<D>(r1, nt) + 4 * tq),
                     "r"(pack_bf16x2(oacc[nt][2] * i1, oacc[nt][3] * i1))
                     : "memory");
    }
    if (tq == 0) {
      float* lrow = lse + static_cast<size_t>(bh) * N + s;
      if (r0 < F) lrow[static_cast<size_t>(r0) * S] = (m0 + __log2f(l0)) * 0.69314718055994530942f;
      if (r1 < F) lrow[static_cast<size_t>(r1) * S] = (m1 + __log2f(l1)) * 0.69314718055994530942f;
    }
  }
  // 6. the F rows of O, 16 bytes a lane
  __syncwarp();
  for (int u = lane; u < F * U; u += 32) {
    const int f = u / U, c = u % U;
    uint4 val;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                 : "r"(qs + sw<D>(f, c))
                 : "memory");
    *reinterpret_cast<uint4*>(out + head + (static_cast<size_t>(f) * S + s) * D + c * 8) = val;
  }
}

template <int D>
size_t smem_bytes(int32_t F) {
  return static_cast<size_t>(kWarps) * 3 * F * D * 2;
}

template <int D>
tsr_status launch_d(const void* q, const void* k, const void* v, void* out, float* lse, int32_t H,
                    int32_t N, int32_t F, int32_t S, const int8_t* head_kind, int64_t bh_lo,
                    int64_t bh_hi, cudaStream_t stream) {
  // the dynamic shared memory limit, once per device (sized for F = 32)
  static bool attr_done[64] = {false};
  int dev = 0;
  TSR_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    TSR_CUDA(cudaFuncSetAttribute(svg_temporal_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem_bytes<D>(kMaxF))));
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  const float scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
  for (int64_t b0 = bh_lo; b0 < bh_hi; b0 += 65535) {       // grid.y <= 65535
    const int64_t b1 = b0 + 65535 < bh_hi ? b0 + 65535 : bh_hi;
    const dim3 grid(static_cast<unsigned>((S + kWarps - 1) / kWarps), static_cast<unsigned>(b1 - b0));
    svg_temporal_kernel<D><<<grid, kWarps * 32, smem_bytes<D>(F), stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), static_cast<__nv_bfloat16*>(out), lse, head_kind, H,
        N, F, S, b0, scale_log2);
    TSR_CUDA(cudaGetLastError());
  }
  return TSR_OK;
}

}  // namespace

bool svg_temporal_eligible(int32_t F, int32_t R, int32_t d) {
  return R == 0 && F >= 1 && F <= kMaxF && (d == 64 || d == 128);
}

tsr_status launch_svg_temporal(const void* q, const void* k, const void* v, void* out, float* lse,
                               int32_t H, int32_t N, int32_t d, int32_t F, int32_t S,
                               const int8_t* head_kind, int64_t bh_lo, int64_t bh_hi,
                               cudaStream_t stream) {
  if (bh_hi <= bh_lo || S <= 0) return TSR_OK;
  if (!svg_temporal_eligible(F, 0, d) || static_cast<int64_t>(F) * S != N)
    return fail(TSR_ERR_INTERNAL, "temporal block shape");
  if (d == 128) return launch_d<128>(q, k, v, out, lse, H, N, F, S, head_kind, bh_lo, bh_hi, stream);
  return launch_d<64>(q, k, v, out, lse, H, N, F, S, head_kind, bh_lo, bh_hi, stream);
}

}  // namespace tsr
