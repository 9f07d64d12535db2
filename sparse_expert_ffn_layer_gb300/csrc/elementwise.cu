// Bandwidth kernels around the expert GEMMs: clearing, the slot-ordered copy of the token
// rows, the fp32 -> output conversion, the standalone gate-weighted combine, and the
// bounded-wait self test.  Grids are sized in
// multiples of the SM count and use 16-byte accesses where the row length allows.
#include "launch.h"

namespace moe {
namespace {

int grid_for(size_t work, int per_block) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  size_t blocks = (work + per_block - 1) / per_block;
  size_t cap = (size_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

__global__ void zero_f32_kernel(float* __restrict__ p, size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t n4 = n / 4;
  float4* p4 = reinterpret_cast<float4*>(p);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride)
    p4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (size_t i = n4 * 4 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = 0.f;
}

// Rows of tokens none of whose assignments were kept become zero (standard top-1 output).
__global__ void zero_dropped_rows_kernel(const int32_t* __restrict__ slot_of, int T, int k,
                                         size_t row_bytes, uint8_t* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    bool any = false;
    for (int j = 0; j < k; ++j) any |= slot_of[(size_t)t * k + j] >= 0;
    if (any) continue;
    uint4* row = reinterpret_cast<uint4*>(out + (size_t)t * row_bytes);
    for (size_t c = lane; c < row_bytes / 16; c += 32) row[c] = make_uint4(0u, 0u, 0u, 0u);
  }
}

template <typename Tout>
__device__ __forceinline__ Tout from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }

template <typename Tv>
__device__ __forceinline__ float as_f32(Tv v);
template <>
__device__ __forceinline__ float as_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float as_f32<__half>(__half v) { return __half2float(v); }

// out = acc32 (+ r32), rounded once; four elements per thread step.
template <typename Tout>
__global__ void finalize_kernel(const float* __restrict__ acc32, const float* __restrict__ r32,
                                size_t n, Tout* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n / 4; i += stride) {
    float4 v = reinterpret_cast<const float4*>(acc32)[i];
    if (r32) {
      float4 r = reinterpret_cast<const float4*>(r32)[i];
      v.x += r.x; v.y += r.y; v.z += r.z; v.w += r.w;
    }
    out[4 * i + 0] = from_f32<Tout>(v.x);
    out[4 * i + 1] = from_f32<Tout>(v.y);
    out[4 * i + 2] = from_f32<Tout>(v.z);
    out[4 * i + 3] = from_f32<Tout>(v.w);
  }
}

// out[t] = sum_j [slot >= 0] w_j expert_out[slot] (+ residual_in[t]); one warp per token row.
// Each lane handles V consecutive columns with 16-byte accesses (V = 8 halves or 4 floats;
// V = 1 where the row length does not allow it).
template <typename T_, int V>
__global__ void combine_kernel(const T_* __restrict__ eo, const int32_t* __restrict__ slot_of,
                               const float* __restrict__ topk_w, const T_* __restrict__ res,
                               int T, int d, int k, T_* __restrict__ out) {
  struct alignas(V * sizeof(T_)) Vec { T_ v[V]; };
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    int s[2];
    float w[2];
    for (int j = 0; j < k; ++j) {
      s[j] = slot_of[(size_t)t * k + j];
      w[j] = topk_w[(size_t)t * k + j];
    }
    for (int c = lane * V; c < d; c += 32 * V) {
      float acc[V];
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = 0.f;
      for (int j = 0; j < k; ++j) {
        if (s[j] < 0) continue;
        const Vec e = *reinterpret_cast<const Vec*>(eo + (size_t)s[j] * d + c);
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] += w[j] * as_f32<T_>(e.v[q]);
      }
      if (res) {
        const Vec r = *reinterpret_cast<const Vec*>(res + (size_t)t * d + c);
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] += as_f32<T_>(r.v[q]);
      }
      Vec o;
#pragma unroll
      for (int q = 0; q < V; ++q) o.v[q] = from_f32<T_>(acc[q]);
      *reinterpret_cast<Vec*>(out + (size_t)t * d + c) = o;
    }
  }
}

// Slot-ordered copy of the dispatched token rows: Xg[s, :] = X[perm[s], :] for every kept slot
// s < min(offsets[E], S_bound), a warp per row with 16-byte accesses.  A perm entry outside
// [0, T) records MOE_ERR_DEVICE_BOUNDS and gives a zero row.
__global__ void gather_rows_kernel(const uint4* __restrict__ X, const int32_t* __restrict__ perm,
                                   const int32_t* __restrict__ offsets, int E, int S_bound, int T,
                                   int row_u4, uint4* __restrict__ Xg, int* status) {
  pdl_wait();
  pdl_trigger();
  const int S = min(max(offsets[E], 0), S_bound);
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int s = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; s < S; s += warps) {
    const int t = perm[s];
    uint4* dst = Xg + (size_t)s * row_u4;
    if ((unsigned)t >= (unsigned)T) {
      if (lane == 0) record_status(status, kErrBounds);
      for (int c = lane; c < row_u4; c += 32) dst[c] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const uint4* src = X + (size_t)t * row_u4;
    for (int c = lane; c < row_u4; c += 32) dst[c] = src[c];
  }
}

__global__ void selftest_wait_kernel(int* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives on `bar`: the wait must give up and record the timeout
    mbar_wait_bounded(&bar, 0, &abort_flag, status, timeout_ns);
  }
  __syncthreads();
}

// Split-K reduction of the first GEMM: sum the chunks in order, GeLU, round to f16.  It lets
// the second GEMM launch before waiting for the first: that GEMM's weight loads depend on
// nothing this chain writes, and it waits for this kernel before it reads H.
__global__ void splitk_reduce1_kernel(const GemmArgs g, int S_max, int T_res, int f, int f_res) {
  pdl_trigger();
  pdl_wait();
  const int S = g.offsets[g.E];
  const size_t n = (size_t)(S_max + T_res) * g.part_cols;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < n; q += stride) {
    const int prow = (int)(q / g.part_cols), c = (int)(q % g.part_cols);
    const bool res = prow >= S_max;
    const int row = res ? prow - S_max : prow;
    if (res ? c >= f_res : (c >= f || row >= S)) continue;
    float v = 0.f;
    for (int ks = 0; ks < g.ksplit; ++ks) v += g.partial[((size_t)ks * g.part_rows + prow) * g.part_cols + c];
    const __half h = __float2half_rn(gelu_tanh(v));
    if (res) g.hres_out[(size_t)row * g.ldhres + c] = h;
    else g.h_out[(size_t)row * g.ldh + c] = h;
  }
}

// Split-K reduction of the second GEMM, then the combine.  At decode sizes its time is the
// latency of its loads: four threads (a quad of lanes) share four adjacent columns of one
// partial row, thread p sums chunks p, p + 4, p + 8, ... in ascending order with 16-byte loads
// (all independent, so they are in flight together, beside the slot's token and gate weight),
// and the quad then adds (s0 + s1) + (s2 + s3) (each pair added in the same order by both lanes
// that form it), so every run gives the same bits.
__global__ void splitk_reduce2_kernel(const GemmArgs g, int S_max, int T_res, int d) {
  pdl_wait();
  pdl_trigger();
  const int S = min(max(g.offsets[g.E], 0), S_max);
  const int cols4 = d / 4;
  const size_t n = (size_t)(S_max + T_res) * cols4;
  const int p = threadIdx.x & 3;
  // a warp takes eight quads per step; the loop bound is the same for the whole warp, so every
  // shuffle below has all 32 lanes
  const size_t gw = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const size_t nw = (size_t)gridDim.x * blockDim.x / 32;
  for (size_t qb = gw * 8; qb < n; qb += nw * 8) {
    const size_t q = qb + (threadIdx.x & 31) / 4;
    const int prow = (int)(q / cols4), c = (int)(q % cols4) * 4;
    const bool res = prow >= S_max;
    const int row = res ? prow - S_max : prow;
    const bool live = q < n && (res || row < S);
    const int nks = g.ksplit;
    // the slot's token and gate weight first, so that their loads overlap the partial sums'
    int tok = 0;
    float w = 1.0f;
    const bool scatter = live && !res && g.mode != kModeExpertOut;
    if (scatter) {
      tok = g.perm[row];
      w = g.slot_w[row];
    }
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
      const float* base = g.partial + (size_t)prow * g.part_cols + c;
      const size_t ks_stride = (size_t)g.part_rows * g.part_cols;
#pragma unroll 4
      for (int ks = p; ks < nks; ks += 4) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(base + (size_t)ks * ks_stride));
        v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
      }
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
      v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
      v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
      v.w += __shfl_xor_sync(0xffffffffu, v.w, o);
    }
    if (!live || p != 0) continue;
    if (res) {
      __half* o = g.out + (size_t)row * g.ldo + c;
      if (g.mode == kModeSum) {
        red_add_f16x2(o, __floats2half2_rn(v.x, v.y));
        red_add_f16x2(o + 2, __floats2half2_rn(v.z, v.w));
      } else {
        *reinterpret_cast<float4*>(g.r32 + (size_t)row * g.ldo + c) = v;
      }
    } else if (g.mode == kModeExpertOut) {
      __half2* o = reinterpret_cast<__half2*>(g.out + (size_t)row * g.ldo + c);
      o[0] = __floats2half2_rn(v.x, v.y);
      o[1] = __floats2half2_rn(v.z, v.w);
    } else {
      if ((unsigned)tok >= (unsigned)g.n_tokens) {
        record_status(g.status, kErrBounds);
        continue;
      }
      __half* o = g.out + (size_t)tok * g.ldo + c;
      if (g.mode == kModeDirect) {
        reinterpret_cast<__half2*>(o)[0] = __floats2half2_rn(w * v.x, w * v.y);
        reinterpret_cast<__half2*>(o)[1] = __floats2half2_rn(w * v.z, w * v.w);
      } else if (g.mode == kModeSum) {
        red_add_f16x2(o, __floats2half2_rn(w * v.x, w * v.y));
        red_add_f16x2(o + 2, __floats2half2_rn(w * v.z, w * v.w));
      } else {
        float* a32 = g.acc32 + (size_t)tok * g.ldo + c;
        red_add_f32(a32, w * v.x);
        red_add_f32(a32 + 1, w * v.y);
        red_add_f32(a32 + 2, w * v.z);
        red_add_f32(a32 + 3, w * v.w);
      }
    }
  }
}

}  // namespace

cudaError_t launch_splitk_reduce1(const GemmArgs& g, int S_max, int T_res, int f, int f_res,
                                  cudaStream_t s, bool pdl) {
  const size_t n = (size_t)(S_max + T_res) * g.part_cols;
  return launch_k(splitk_reduce1_kernel, grid_for(n, 256), 256, 0, s, pdl, g, S_max, T_res, f,
                  f_res);
}

cudaError_t launch_splitk_reduce2(const GemmArgs& g, int S_max, int T_res, int d, cudaStream_t s,
                                  bool pdl) {
  const size_t n = (size_t)(S_max + T_res) * d;
  return launch_k(splitk_reduce2_kernel, grid_for(n, 256), 256, 0, s, pdl, g, S_max, T_res, d);
}

cudaError_t launch_gather_rows(const void* X, const int32_t* perm, const int32_t* offsets, int E,
                               int S_bound, int T, int row_bytes, void* Xg, int* status,
                               cudaStream_t s, bool pdl) {
  // a warp per row, at most 8 CTAs of 128 threads per SM
  return launch_k(gather_rows_kernel, grid_for((size_t)S_bound * 32, 128), 128, 0, s, pdl,
                  static_cast<const uint4*>(X), perm, offsets, E, S_bound, T, row_bytes / 16,
                  static_cast<uint4*>(Xg), status);
}

cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t s) {
  MOE_LAUNCH(launch_k(zero_f32_kernel, grid_for(n / 4 + 1, 256), 256, 0, s, false, p, n));
  return cudaGetLastError();
}

cudaError_t launch_zero_dropped_rows(const int32_t* slot_of, int T, int k, int d, int dtype_f16,
                                     void* out, cudaStream_t s) {
  const size_t row_bytes = (size_t)d * (dtype_f16 ? 2 : 4);
  MOE_LAUNCH(launch_k(zero_dropped_rows_kernel, grid_for((size_t)T * 32, 256), 256, 0, s, false,
                      slot_of, T, k, row_bytes, static_cast<uint8_t*>(out)));
  return cudaGetLastError();
}

cudaError_t launch_finalize(const float* acc32, const float* r32, int T, int d, int dtype_f16,
                            void* out, cudaStream_t s, bool pdl) {
  const size_t n = (size_t)T * d;
  const int g = grid_for(n / 4, 256);
  if (dtype_f16)
    return launch_k(finalize_kernel<__half>, g, 256, 0, s, pdl, acc32, r32, n,
                    static_cast<__half*>(out));
  return launch_k(finalize_kernel<float>, g, 256, 0, s, pdl, acc32, r32, n, static_cast<float*>(out));
}

cudaError_t launch_combine(const void* expert_out, const int32_t* slot_of, const float* topk_w,
                           const void* residual_in, int dtype_f16, int T, int d, int k, void* out,
                           cudaStream_t s) {
  const int g = grid_for((size_t)T * 32, 256);
  const bool a16 = ((reinterpret_cast<uintptr_t>(expert_out) | reinterpret_cast<uintptr_t>(out) |
                     reinterpret_cast<uintptr_t>(residual_in)) & 15) == 0;
  if (dtype_f16) {
    const __half* eo = static_cast<const __half*>(expert_out);
    const __half* ri = static_cast<const __half*>(residual_in);
    __half* o = static_cast<__half*>(out);
    if (d % 8 == 0 && a16)
      MOE_LAUNCH(launch_k(combine_kernel<__half, 8>, g, 256, 0, s, false, eo, slot_of, topk_w, ri, T,
                          d, k, o));
    else
      MOE_LAUNCH(launch_k(combine_kernel<__half, 1>, g, 256, 0, s, false, eo, slot_of, topk_w, ri, T,
                          d, k, o));
  } else {
    const float* eo = static_cast<const float*>(expert_out);
    const float* ri = static_cast<const float*>(residual_in);
    float* o = static_cast<float*>(out);
    if (d % 4 == 0 && a16)
      MOE_LAUNCH(launch_k(combine_kernel<float, 4>, g, 256, 0, s, false, eo, slot_of, topk_w, ri, T,
                          d, k, o));
    else
      MOE_LAUNCH(launch_k(combine_kernel<float, 1>, g, 256, 0, s, false, eo, slot_of, topk_w, ri, T,
                          d, k, o));
  }
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int* status, uint64_t timeout_ns, cudaStream_t s) {
  MOE_LAUNCH(launch_k(selftest_wait_kernel, 1, 32, 0, s, false, status, timeout_ns));
  return cudaGetLastError();
}

}  // namespace moe
