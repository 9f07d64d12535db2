// Fused router for decode-sized batches: gate logits, softmax / top-k and the capacity
// dispatch of a whole batch of T <= 64 tokens in one launch.
//
// What it computes is exactly what the three separate kernels compute (gate.cu, dispatch.cu):
// the fp32 logit chain acc = fmaf(x[t,i], Wg[i,e], acc) in ascending i from +0 (gating
// function: DeepSpeed-MoE review, "MoE based NLG Model Architecture"), top-k on the logits
// with ties to the lower index and the softmax weights (topk.cuh), then the token-order
// capacity rule with compact slots (C = ceil(cf T / E), a reading: the pages give no
// per-expert token capacity).
//
// Shape of the work.  At decode sizes the gate is latency-bound: T * E chains of d dependent
// FMAs and a Wg read of d * E * 4 bytes.  Each CTA owns 4 experts x 64 tokens (one chain per
// thread) and streams its Wg columns and the batch's token rows through a four-deep cp.async
// ring, so E / 4 CTAs (32 at E = 128) pull Wg in parallel.  The last CTA to finish (a counter in the
// workspace, cleared by the caller before the launch and by that CTA after use) then routes
// the whole batch: a warp per token for softmax / top-k, then the dispatch of the T * k <= 128
// assignments by one block (per-expert counts and ranks counted directly over the assignment
// list, no atomics).
#include <algorithm>

#include "launch.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kRExp = 4;            // experts per CTA
constexpr int kRTok = 64;           // tokens per CTA (T <= 64: one row of CTAs)
constexpr int kRKC = 128;           // shared-dimension chunk
constexpr int kRStages = 4;         // cp.async ring depth
constexpr int kRXPitch = kRKC + 8;  // halves per staged token row: the 16-byte pad spreads the
                                    // eight rows a warp reads over distinct banks
constexpr int kRThreads = kRExp * kRTok;
constexpr int kRTokPerWarp = 32 / kRExp;
constexpr size_t kRWBytes = (size_t)kRKC * kRExp * 4;

// Shared memory of a launch: the ring (Wg chunk and the batch's token rows per stage), and at
// least the routing scratch the last CTA reuses it for.
// Token rows per stage: the batch's, rounded up to whole warps (a warp's threads read the rows
// of its eight tokens, valid or not; only valid tokens' results are stored).
__host__ __device__ inline size_t route_stage_bytes(int nT) {
  const int rows = (nT + kRTokPerWarp - 1) / kRTokPerWarp * kRTokPerWarp;
  return kRWBytes + (size_t)rows * kRXPitch * 2;
}
inline size_t route_smem_bytes(int nT, int E) {
  const size_t ring = kRStages * route_stage_bytes(nT);
  const size_t scratch = (size_t)(256 + 2 * E + kRThreads / 32) * 4;
  return ring > scratch ? ring : scratch;
}

struct RouteArgs {
  const __half* x;       // [T, d]
  const float* Wg;       // [d, E]
  int T, d, E, k, C;
  float* logits;         // [T, E]
  int32_t* topk_idx;     // [T, k]
  float* topk_w;         // [T, k]
  int32_t* counts_raw;   // [E]
  int32_t* kept;         // [E]
  int32_t* offsets;      // [E + 1]
  int32_t* perm;         // [min(T k, E C)]
  int32_t* slot_of;      // [T, k]
  float* slot_w;         // [min(T k, E C)]
  unsigned int* counter; // zero at launch
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Loads through L2 only: the logits of other CTAs are read after their release.
struct L2Load {
  __device__ __forceinline__ float operator()(const float* p) const { return __ldcg(p); }
};

// Needs f16 tokens, d % 128 == 0, E % 4 == 0, 16-byte aligned x and Wg, T <= 64.
__global__ void __launch_bounds__(kRThreads) gate_route_small_kernel(const RouteArgs a) {
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ int s_last;
  const int ee = threadIdx.x & (kRExp - 1), tt = threadIdx.x / kRExp;
  const int e0 = blockIdx.x * kRExp, t0 = blockIdx.y * kRTok;
  const int nT = min(kRTok, a.T - t0);
  const int nch = a.d / kRKC;
  const size_t stage_bytes = route_stage_bytes(min(kRTok, a.T));
  // a warp holds tokens 8w .. 8w+7: warps past the batch's last token only help load
  const bool computes = (tt & ~(kRTokPerWarp - 1)) < nT;

  auto issue = [&](int c) {
    uint8_t* base = sm + (size_t)(c % kRStages) * stage_bytes;
    const int i0 = c * kRKC;
    // Wg rows i0 .. i0+127, experts e0 .. e0+3: one 16-byte piece per row
    for (int row = threadIdx.x; row < kRKC; row += kRThreads)
      cp_async16(base + row * (kRExp * 4), a.Wg + (size_t)(i0 + row) * a.E + e0);
    uint8_t* xb = base + kRWBytes;     // the valid token rows, 16 pieces each
    for (int q = threadIdx.x; q < nT * (kRKC / 8); q += kRThreads) {
      const int r = q / (kRKC / 8), col = (q % (kRKC / 8)) * 8;
      cp_async16(xb + (size_t)(r * kRXPitch + col) * 2, a.x + (size_t)(t0 + r) * a.d + i0 + col);
    }
  };

#pragma unroll
  for (int c = 0; c < kRStages - 1; ++c) {
    if (c < nch) issue(c);
    cp_async_commit();
  }
  float acc = 0.0f;
  for (int c = 0; c < nch; ++c) {
    if (c + kRStages - 1 < nch) issue(c + kRStages - 1);
    cp_async_commit();
    cp_async_wait<kRStages - 1>();
    __syncthreads();
    const uint8_t* base = sm + (size_t)(c % kRStages) * stage_bytes;
    const float* ws = reinterpret_cast<const float*>(base) + ee;
    const __half* xs = reinterpret_cast<const __half*>(base + kRWBytes) + tt * kRXPitch;
    if (computes) {
#pragma unroll 4
      for (int i = 0; i < kRKC; i += 8) {             // ascending i
        const uint4 raw = *reinterpret_cast<const uint4*>(xs + i);
        const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __half22float2(h[q]);      // exact widening
          acc = __fmaf_rn(f.x, ws[(i + 2 * q) * kRExp], acc);
          acc = __fmaf_rn(f.y, ws[(i + 2 * q + 1) * kRExp], acc);
        }
      }
    }
    __syncthreads();                                  // the slot may be refilled next
  }
  cp_async_wait<0>();
  if (tt < nT) a.logits[(size_t)(t0 + tt) * a.E + e0 + ee] = acc;

  // ---------------------------------------------------------------- last CTA: routing
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.counter, 1u) == gridDim.x * gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  constexpr int kWarps = kRThreads / 32;
  const int n = a.T * a.k;                            // <= 128 assignments
  int32_t* s_idx = reinterpret_cast<int32_t*>(sm);    // the ring is free now
  float* s_w = reinterpret_cast<float*>(s_idx + 128);
  int32_t* s_cnt = reinterpret_cast<int32_t*>(s_w + 128);   // [E]
  int32_t* s_off = s_cnt + a.E;                             // [E]
  int32_t* s_wsum = s_off + a.E;                            // [kWarps]

  for (int tok = w; tok < a.T; tok += kWarps) {
    const TopK r = softmax_topk_warp(a.logits + (size_t)tok * a.E, a.E, a.k, lane, L2Load(),
                                     nullptr, nullptr);
    if (lane == 0) {
      for (int j = 0; j < a.k; ++j) {
        const int q = tok * a.k + j;
        s_idx[q] = r.idx[j];
        s_w[q] = r.w[j];
        a.topk_idx[q] = r.idx[j];
        a.topk_w[q] = r.w[j];
      }
    }
  }
  __syncthreads();
  // assignments per expert, counted directly over the <= 128 assignments (no atomics; an index
  // outside [0, E) from NaN logits matches no expert)
  for (int e = threadIdx.x; e < a.E; e += kRThreads) {
    int c = 0;
    for (int q = 0; q < n; ++q) c += s_idx[q] == e;
    s_cnt[e] = c;
  }
  __syncthreads();
  // kept = min(count, C) and its exclusive scan; thread th owns a run of experts
  const int per = (a.E + kRThreads - 1) / kRThreads;
  const int lo = min(a.E, (int)threadIdx.x * per), hi = min(a.E, lo + per);
  int local = 0;
  for (int e = lo; e < hi; ++e) local += min(s_cnt[e], a.C);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int v = lane < kWarps ? s_wsum[lane] : 0;
    int sc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, sc, o);
      if (lane >= o) sc += u;
    }
    if (lane < kWarps) s_wsum[lane] = sc - v;
  }
  __syncthreads();
  int run = s_wsum[w] + incl - local;
  for (int e = lo; e < hi; ++e) {
    const int kp = min(s_cnt[e], a.C);
    s_off[e] = run;
    a.offsets[e] = run;
    a.counts_raw[e] = s_cnt[e];
    a.kept[e] = kp;
    run += kp;
  }
  if (lo < hi && hi == a.E) a.offsets[a.E] = run;
  __syncthreads();
  // rank of an assignment = earlier assignments (token-major order) to the same expert
  for (int q = threadIdx.x; q < n; q += kRThreads) {
    const int e = s_idx[q];
    int r = 0;
    for (int p = 0; p < q; ++p) r += s_idx[p] == e;
    int slot = -1;
    if ((unsigned)e < (unsigned)a.E && r < a.C) {
      slot = s_off[e] + r;
      a.perm[slot] = q / a.k;
      a.slot_w[slot] = s_w[q];
    }
    a.slot_of[q] = slot;
  }
  if (threadIdx.x == 0) *a.counter = 0u;              // ready for the next launch
}

}  // namespace

bool gate_route_small_ok(int T, int d, int E, const void* x, const void* Wg) {
  return T >= 1 && T <= kRTok && d % kRKC == 0 && E % kRExp == 0 && E <= 1024 &&
         (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (reinterpret_cast<uintptr_t>(Wg) & 15) == 0;
}

cudaError_t launch_gate_route_small(const __half* x, const float* Wg, int T, int d, int E, int k,
                                    int C, float* logits, int32_t* topk_idx, float* topk_w,
                                    int32_t* counts_raw, int32_t* kept, int32_t* offsets,
                                    int32_t* perm, int32_t* slot_of, float* slot_w,
                                    unsigned int* counter, cudaStream_t s) {
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(gate_route_small_kernel));
  if (err != cudaSuccess) return err;
  RouteArgs a{x, Wg, T, d, E, k, C, logits, topk_idx, topk_w, counts_raw, kept, offsets, perm,
              slot_of, slot_w, counter};
  dim3 grid(E / kRExp, (T + kRTok - 1) / kRTok);
  return launch_k(gate_route_small_kernel, grid, kRThreads, route_smem_bytes(std::min(T, kRTok), E),
                  s, false, a);
}

}  // namespace moe
