// fp32 expert FFN on the CUDA cores, for float32 layers (small shapes such as d = 64).
//
// Same grouping, GeLU and combine rules as the tensor-core path: block (c, g, r) computes a
// 32-row x 64-column tile of group g (experts in slot order, then the residual group of all
// tokens), rows 32 r .. 32 r + 31 of the group, with fp32 fused multiply-adds.
#include "launch.h"

namespace moe {
namespace {

constexpr int kR = 32, kC = 64, kKC = 32;

template <int kStage>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtArgs a) {
  __shared__ float xs[kR][kKC + 1];
  __shared__ float ws[kKC][kC];
  const int g = blockIdx.y;
  const bool res = g == a.E;
  int rows, row0;
  if (res) {
    rows = a.T;
    row0 = 0;
  } else {
    // slot range of expert g, clamped to [0, S_bound): offsets that run past the caller's
    // S_max leave the rows beyond it uncomputed instead of writing past H or the output
    row0 = min(max(a.offsets[g], 0), a.S_bound);
    rows = min(max(a.offsets[g + 1], row0), a.S_bound) - row0;
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0 &&
        (row0 != a.offsets[g] || row0 + rows != a.offsets[g + 1]))
      record_status(a.status, kErrBounds);
  }
  const int r0 = blockIdx.z * kR;
  if (r0 >= rows) return;
  const int n_cols = kStage == 1 ? (res ? a.f_res : a.f) : a.d;
  const int c0 = blockIdx.x * kC;
  if (c0 >= n_cols) return;
  const int K = kStage == 1 ? a.d : (res ? a.f_res : a.f);
  const float* W = kStage == 1 ? (res ? a.Wr1 : a.W1 + (size_t)g * a.d * a.f)
                               : (res ? a.Wr2 : a.W2 + (size_t)g * a.f * a.d);
  const int ldw = n_cols;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;   // 64 columns x 4 row lanes
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kKC) {
    const int kc = min(kKC, K - k0);
    for (int q = threadIdx.x; q < kR * kKC; q += 256) {
      const int rr = q / kKC, kk = q % kKC;
      const int r = r0 + rr;
      float v = 0.f;
      if (r < rows && kk < kc) {
        if (kStage == 1) {
          const int tok = res ? r : a.perm[row0 + r];
          // a token index outside [0, T) reads as a zero row and records the error
          if ((unsigned)tok < (unsigned)a.T) v = a.x[(size_t)tok * a.d + k0 + kk];
          else record_status(a.status, kErrBounds);
        } else {
          v = res ? a.Hres[(size_t)r * a.f_res + k0 + kk] : a.H[(size_t)(row0 + r) * a.f + k0 + kk];
        }
      }
      xs[rr][kk] = v;
    }
    for (int q = threadIdx.x; q < kKC * kC; q += 256) {
      const int kk = q / kC, cc = q % kC;
      ws[kk][cc] = (kk < kc && c0 + cc < n_cols) ? W[(size_t)(k0 + kk) * ldw + c0 + cc] : 0.f;
    }
    __syncthreads();
    for (int kk = 0; kk < kc; ++kk) {
      const float w = ws[kk][tx];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = __fmaf_rn(xs[ty + 4 * q][kk], w, acc[q]);
    }
    __syncthreads();
  }
  const int c = c0 + tx;
  if (c >= n_cols) return;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int r = r0 + ty + 4 * q;
    if (r >= rows) continue;
    if (kStage == 1) {
      const float h = gelu_tanh(acc[q]);
      if (res) a.Hres[(size_t)r * a.f_res + c] = h;
      else a.H[(size_t)(row0 + r) * a.f + c] = h;
    } else if (res) {
      if (a.mode == kModeSum) red_add_f32(a.out + (size_t)r * a.d + c, acc[q]);
      else a.r32[(size_t)r * a.d + c] = acc[q];
    } else {
      const int slot = row0 + r;
      if (a.mode == kModeExpertOut) {
        a.out[(size_t)slot * a.d + c] = acc[q];
      } else {
        const int tok = a.perm[slot];
        const float w = a.slot_w[slot];
        if (a.mode == kModeDirect) a.out[(size_t)tok * a.d + c] = w * acc[q];
        else if (a.mode == kModeSum) red_add_f32(a.out + (size_t)tok * a.d + c, w * acc[q]);
        else red_add_f32(a.acc32 + (size_t)tok * a.d + c, w * acc[q]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_simt_ffn1(const SimtArgs& a, int rows_bound, cudaStream_t s) {
  const int cols = max(a.f, a.Wr1 ? a.f_res : 0);
  dim3 grid((cols + kC - 1) / kC, a.E + (a.Wr1 ? 1 : 0), (rows_bound + kR - 1) / kR);
  MOE_LAUNCH(launch_k(simt_gemm_kernel<1>, grid, 256, 0, s, false, a));
  return cudaGetLastError();
}

cudaError_t launch_simt_ffn2(const SimtArgs& a, int rows_bound, cudaStream_t s) {
  dim3 grid((a.d + kC - 1) / kC, a.E + (a.Wr2 ? 1 : 0), (rows_bound + kR - 1) / kR);
  MOE_LAUNCH(launch_k(simt_gemm_kernel<2>, grid, 256, 0, s, false, a));
  return cudaGetLastError();
}

}  // namespace moe
