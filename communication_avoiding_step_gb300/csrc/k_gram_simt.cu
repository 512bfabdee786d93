// Step a3 on CUDA cores: G_{j,t} = Y_j Y_t^T from BF16 Y with FP32 FMA accumulation.
//
// Paper: Mixed-Precision Communication-Avoiding SGD for Generalized Linear Models on
// GPUs (abstract): the Gram matrix is formed from low-precision inputs with
// high-precision accumulation.  Only the blocks the inner recurrence reads (t < j),
// plus the diagonal blocks on request, are computed and stored, in the packed
// block-lower layout of include/casgd.h.
//
// This kernel serves narrow feature counts (n of a few tens), where the step is bound
// by writing G to HBM rather than by arithmetic, and any shape the tensor-core kernel
// does not take.  A CTA computes one 64x64 tile of the S x S matrix with 256 threads,
// 4x4 outputs each; K is staged through shared memory 32 columns at a time as FP32.
#include "casgd_internal.cuh"

namespace casgd {

namespace {

constexpr int kTile = 64;
constexpr int kKC = 32;

__global__ void __launch_bounds__(256) gram_simt_kernel(const uint16_t* __restrict__ Y,
                                                        int64_t S, int64_t ldY, int b,
                                                        bool diag, bool g_bf16,
                                                        float* __restrict__ G) {
  const int64_t R0 = (int64_t)blockIdx.y * kTile;
  const int64_t C0 = (int64_t)blockIdx.x * kTile;
  if (R0 >= S || C0 >= S) return;
  const int64_t last_row = (R0 + kTile - 1 < S) ? R0 + kTile - 1 : S - 1;
  const int64_t jmax = last_row / b, tmin = C0 / b;
  if (jmax < tmin || (jmax == tmin && !diag)) return;  // tile lies above the needed blocks

  __shared__ float As[kKC][kTile + 4];
  __shared__ float Bs[kKC][kTile + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  float acc[4][4] = {};

  // loader: thread -> (row tid/4, 8-column vector tid%4) of the 64 x 32 slab
  const int lr = tid >> 2, lv = tid & 3;
  for (int64_t k0 = 0; k0 < ldY; k0 += kKC) {
    const int64_t kc = k0 + lv * 8;
    uint4 qa = make_uint4(0, 0, 0, 0), qb = make_uint4(0, 0, 0, 0);
    if (kc < ldY) {
      if (R0 + lr < S) qa = __ldg(reinterpret_cast<const uint4*>(Y + (R0 + lr) * ldY + kc));
      if (C0 + lr < S) qb = __ldg(reinterpret_cast<const uint4*>(Y + (C0 + lr) * ldY + kc));
    }
    const uint32_t pa[4] = {qa.x, qa.y, qa.z, qa.w};
    const uint32_t pb[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      As[lv * 8 + 2 * h][lr] = bf16_bits_to_float(pa[h] & 0xFFFFu);
      As[lv * 8 + 2 * h + 1][lr] = bf16_bits_to_float(pa[h] >> 16);
      Bs[lv * 8 + 2 * h][lr] = bf16_bits_to_float(pb[h] & 0xFFFFu);
      Bs[lv * 8 + 2 * h + 1][lr] = bf16_bits_to_float(pb[h] >> 16);
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKC; ++kk) {
      const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = As[kk][ty + 16 * i];
        acc[i][0] = fmaf(a, bv.x, acc[i][0]);
        acc[i][1] = fmaf(a, bv.y, acc[i][1]);
        acc[i][2] = fmaf(a, bv.z, acc[i][2]);
        acc[i][3] = fmaf(a, bv.w, acc[i][3]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t p = R0 + ty + 16 * i;
    if (p >= S) continue;
    const int64_t jb = p / b;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t q = C0 + tx * 4 + e;
      if (q >= S) continue;
      const int64_t tb = q / b;
      if (tb > jb || (tb == jb && !diag)) continue;
      G[packed_offset(jb, tb, b, diag) + (p - jb * b) * b + (q - tb * b)] =
          g_bf16 ? round_bf16(acc[i][e]) : acc[i][e];
    }
  }
}

}  // namespace

cudaError_t launch_gram_simt(const uint16_t* Y, int64_t S, int64_t n, int64_t ldY, int b,
                             int s, bool diag, bool g_bf16, float* G, Ctx& c) {
  (void)n;
  (void)s;
  const int64_t T = (S + kTile - 1) / kTile;
  dim3 grid((unsigned)T, (unsigned)T);
  gram_simt_kernel<<<grid, 256, 0, c.stream>>>(Y, S, ldY, b, diag, g_bf16, G);
  ++c.launches;
  return cudaGetLastError();
}

}  // namespace casgd
