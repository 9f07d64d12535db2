// Gate: fp32 logits, softmax and top-k.
//
// Each token reaches its experts through a gating function (DeepSpeed-MoE review, "MoE based
// NLG Model Architecture"); Top2-MoE sends it to two (same review, "Phenomenon2").  The
// logits are the fp32 chain acc = fmaf(x[t,i], Wg[i,e], acc) for i ascending from +0: each
// thread owns whole outputs of a register tile and walks the shared dimension in order, so
// the result is bit-identical to any IEEE evaluation of that chain and routing is exact.
#include "launch.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kTT = 64;   // tokens per block tile (scalar kernel)
constexpr int kTE = 64;   // experts per block tile
constexpr int kKC = 32;   // shared-dimension chunk staged in shared memory
constexpr int kXP = kKC + 4;  // padded row of the token tile (16-byte aligned rows)

// Token tile of the vector kernel (64, 32 or 16 tokens: 256, 128 or 64 threads): the largest
// that still gives about 0.8 CTAs per SM, since a batch of a few hundred tokens leaves most SMs
// idle with 64-token tiles (measured: T = 512 gate 44 -> 32 us with 32-token tiles; T = 4096
// keeps 64).
int sm_count() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    sms = n > 0 ? n : 1;
  }
  return sms;
}

int vec_tile_tokens(int T, int E) {
  const long long etiles = (E + kTE - 1) / kTE;
  for (int t = 64; t > 16; t /= 2)
    if ((T + t - 1) / t * etiles * 5 >= 4LL * sm_count()) return t;
  return 16;
}

template <typename Tin>
struct XChunk;  // one thread's share of a 64 x 32 token chunk: 8 consecutive values of a row

template <>
struct XChunk<__half> {
  uint4 raw;
  __device__ __forceinline__ void load(const __half* p) { raw = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void zero() { raw = make_uint4(0u, 0u, 0u, 0u); }
  __device__ __forceinline__ void to_f32(float (&v)[8]) const {
    const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float2 f = __half22float2(h[q]);      // exact widening
      v[2 * q] = f.x;
      v[2 * q + 1] = f.y;
    }
  }
};

template <>
struct XChunk<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = *reinterpret_cast<const float4*>(p);
    b = *reinterpret_cast<const float4*>(p + 4);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void to_f32(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// logits[T, E] = x[T, d] . Wg[d, E]; 256 threads, 4 x 4 outputs per thread.  The next chunk
// is fetched into registers while the current one is multiplied (double-buffered tiles).
// Vector path: d % 8 == 0 and E % 4 == 0 (16-byte loads); otherwise the scalar kernel below.
template <typename Tin, int kT>
__global__ void __launch_bounds__(kT * 4) gate_logits_kernel(const Tin* __restrict__ x,
                                                            const float* __restrict__ Wg, int T,
                                                            int d, int E,
                                                            float* __restrict__ logits) {
  pdl_trigger();   // the top-k kernel may start its launch; it waits for these logits
  constexpr int kThreadsT = kT * 4;                 // 4 x 4 outputs per thread
  constexpr int kWR = kKC * 16 / kThreadsT;         // Wg rows each thread stages per chunk
  __shared__ __align__(16) float xs[2][kT][kXP];    // token tile: xs[t][i]
  __shared__ __align__(16) float ws[2][kKC][kTE];   // Wg tile: ws[i][e]
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int t0 = blockIdx.x * kT, e0 = blockIdx.y * kTE;
  // loader roles: token row lt, columns lk .. lk+7; Wg rows lw + q * (threads / 16), 4 experts at le
  const int lt = threadIdx.x >> 2, lk = (threadIdx.x & 3) * 8;
  const int lw = threadIdx.x >> 4, le = (threadIdx.x & 15) * 4;
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;

  XChunk<Tin> xr;
  float4 wr[kWR];
  auto fetch = [&](int k0) {
    const int t = t0 + lt;
    const int kc = min(kKC, d - k0);
    if (t < T && lk < kc) xr.load(x + (size_t)t * d + k0 + lk);
    else xr.zero();
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const bool eok = e0 + le < E;
#pragma unroll
    for (int q = 0; q < kWR; ++q) {
      const int row = lw + q * (kThreadsT / 16);
      wr[q] = (eok && row < kc) ? *reinterpret_cast<const float4*>(Wg + (size_t)(k0 + row) * E + e0 + le) : z;
    }
  };
  auto stash = [&](int buf) {
    float v[8];
    xr.to_f32(v);
    *reinterpret_cast<float4*>(&xs[buf][lt][lk]) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(&xs[buf][lt][lk + 4]) = make_float4(v[4], v[5], v[6], v[7]);
#pragma unroll
    for (int q = 0; q < kWR; ++q)
      *reinterpret_cast<float4*>(&ws[buf][lw + q * (kThreadsT / 16)][le]) = wr[q];
  };

  fetch(0);
  stash(0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < d; k0 += kKC) {
    const int kc = min(kKC, d - k0);
    const bool more = k0 + kKC < d;
    if (more) fetch(k0 + kKC);
    auto step = [&](int kk) {                      // one i: 16 chained multiply-adds
      const float4 b = *reinterpret_cast<const float4*>(&ws[buf][kk][tx * 4]);
      const float av[4] = {xs[buf][ty * 4][kk], xs[buf][ty * 4 + 1][kk], xs[buf][ty * 4 + 2][kk],
                           xs[buf][ty * 4 + 3][kk]};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
    };
    if (kc == kKC) {                               // full chunk: straight-line code
#pragma unroll
      for (int kk = 0; kk < kKC; ++kk) step(kk);   // ascending i
    } else {
      for (int kk = 0; kk < kc; ++kk) step(kk);    // ascending i, no padding steps
    }
    if (more) stash(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
    const int e = e0 + tx * 4;
    if (e + 3 < E) {
      *reinterpret_cast<float4*>(logits + (size_t)t * E + e) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (e + j < E) logits[(size_t)t * E + e + j] = acc[i][j];
    }
  }
}

template <typename Tin>
__device__ __forceinline__ float to_f32(Tin v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

// Any d and E: scalar staging, same per-output chain.
template <typename Tin>
__global__ void __launch_bounds__(256) gate_logits_scalar_kernel(const Tin* __restrict__ x,
                                                                 const float* __restrict__ Wg,
                                                                 int T, int d, int E,
                                                                 float* __restrict__ logits) {
  pdl_trigger();   // the top-k kernel may start its launch; it waits for these logits
  __shared__ float xs[kTT][kKC + 1];
  __shared__ __align__(16) float ws[kKC][kTE];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int t0 = blockIdx.x * kTT, e0 = blockIdx.y * kTE;
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.0f;
  for (int k0 = 0; k0 < d; k0 += kKC) {
    const int kc = min(kKC, d - k0);
    for (int q = threadIdx.x; q < kTT * kKC; q += 256) {
      int tt = q / kKC, kk = q % kKC;
      int t = t0 + tt;
      xs[tt][kk] = (t < T && kk < kc) ? to_f32<Tin>(x[(size_t)t * d + k0 + kk]) : 0.0f;
    }
    for (int q = threadIdx.x; q < kTE * kKC; q += 256) {
      int kk = q / kTE, ee = q % kTE;
      int e = e0 + ee;
      ws[kk][ee] = (e < E && kk < kc) ? Wg[(size_t)(k0 + kk) * E + e] : 0.0f;
    }
    __syncthreads();
    for (int kk = 0; kk < kc; ++kk) {
      float av[4] = {xs[ty * 4][kk], xs[ty * 4 + 1][kk], xs[ty * 4 + 2][kk], xs[ty * 4 + 3][kk]};
      float bv[4] = {ws[kk][tx * 4], ws[kk][tx * 4 + 1], ws[kk][tx * 4 + 2], ws[kk][tx * 4 + 3]};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = e0 + tx * 4 + j;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------------------
// Small and medium batches: one thread per expert and M tokens (M independent chains).
// Block = 8 warps x M tokens x 32 experts (lanes); raw Wg and token chunks stream through a
// four-deep cp.async ring, so with few tokens the cost is close to the d dependent
// multiply-adds of one chain instead of a 64-token tile's.
constexpr int kSKC = 64;       // shared-dimension chunk
constexpr int kSStages = 4;    // ring depth
constexpr int kSWarps = 8;     // warps per block; each owns M consecutive tokens
constexpr int kSExp = 32;      // experts per block (one per lane)

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename Tin, int M>
__host__ __device__ constexpr size_t small_slot_bytes() {
  return (size_t)kSKC * kSExp * sizeof(float) + (size_t)kSWarps * M * kSKC * sizeof(Tin);
}

// Eight 16-byte row pieces of a staged token chunk, widened to fp32 (exact).
__device__ __forceinline__ void unpack16(const uint4& u, float* f, const float*) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack16(const uint4& u, float* f, const __half*) {
  const uint32_t r[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&r[q]));
    f[2 * q] = v.x;
    f[2 * q + 1] = v.y;
  }
}

// Needs d % 64 == 0, E % 4 == 0, 16-byte aligned rows.  Warp w owns tokens t0 + w*M .. +M-1,
// lane l expert e0 + l: M independent chains per thread, each in ascending i.
template <typename Tin, int M>
__global__ void __launch_bounds__(256) gate_logits_small_kernel(const Tin* __restrict__ x,
                                                                const float* __restrict__ Wg,
                                                                int T, int d, int E,
                                                                float* __restrict__ logits) {
  pdl_trigger();   // the top-k kernel may start its launch; it waits for these logits
  extern __shared__ __align__(16) uint8_t ssm[];
  constexpr int kTok = kSWarps * M;
  constexpr int kPer = 16 / (int)sizeof(Tin);   // values per 16-byte piece
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e0 = blockIdx.x * kSExp, t0 = blockIdx.y * kTok;
  const int nch = d / kSKC;
  constexpr size_t slot = small_slot_bytes<Tin, M>();
  auto issue = [&](int c) {
    uint8_t* base = ssm + (size_t)(c % kSStages) * slot;
    const int k0 = c * kSKC;
    // Wg rows k0 .. k0+63, experts e0 .. e0+31: 64 x 8 pieces of 16 bytes
    for (int q = threadIdx.x; q < kSKC * (kSExp / 4); q += 256) {
      const int row = q >> 3, col = (q & 7) * 4;
      const int e = e0 + col;
      cp_async16(base + (row * kSExp + col) * 4, Wg + (size_t)(k0 + row) * E + min(e, E - 4),
                 e < E ? 16 : 0);
    }
    // tokens t0 .. t0+kTok-1, columns k0 .. k0+63
    uint8_t* xb = base + (size_t)kSKC * kSExp * 4;
    for (int q = threadIdx.x; q < kTok * (kSKC / kPer); q += 256) {
      const int tt = q / (kSKC / kPer), col = (q % (kSKC / kPer)) * kPer;
      const int t = t0 + tt;
      cp_async16(xb + (tt * kSKC + col) * sizeof(Tin), x + (size_t)min(t, T - 1) * d + k0 + col,
                 t < T ? 16 : 0);
    }
  };
#pragma unroll
  for (int c = 0; c < kSStages - 1; ++c) {
    if (c < nch) issue(c);
    cp_async_commit();
  }
  float acc[M];
#pragma unroll
  for (int j = 0; j < M; ++j) acc[j] = 0.0f;
  for (int c = 0; c < nch; ++c) {
    if (c + kSStages - 1 < nch) issue(c + kSStages - 1);
    cp_async_commit();
    cp_async_wait<kSStages - 1>();
    __syncthreads();
    const uint8_t* base = ssm + (size_t)(c % kSStages) * slot;
    const float* ws = reinterpret_cast<const float*>(base);
    const Tin* xs = reinterpret_cast<const Tin*>(base + (size_t)kSKC * kSExp * 4) + w * M * kSKC;
#pragma unroll 2
    for (int kk = 0; kk < kSKC; kk += kPer) {
      float xv[M][kPer];
#pragma unroll
      for (int j = 0; j < M; ++j)
        unpack16(*reinterpret_cast<const uint4*>(xs + j * kSKC + kk), xv[j], xs);
#pragma unroll
      for (int v = 0; v < kPer; ++v) {             // ascending i
        const float wv = ws[(kk + v) * kSExp + lane];
#pragma unroll
        for (int j = 0; j < M; ++j) acc[j] = __fmaf_rn(xv[j][v], wv, acc[j]);
      }
    }
    __syncthreads();                             // the slot may be refilled next
  }
  cp_async_wait<0>();
  const int e = e0 + lane;
#pragma unroll
  for (int j = 0; j < M; ++j) {
    const int t = t0 + w * M + j;
    if (t < T && e < E) logits[(size_t)t * E + e] = acc[j];
  }
}

// Tokens per warp of the small-batch kernel, 0 where the tiled kernel is used instead: one
// token per warp while that fits one wave of CTAs, two while it fits two waves, else the
// 4x4-per-thread tiled kernel, whose fewer shared-memory reads per multiply-add win once every
// SM is busy.  Measured gate times (350M+MoE-128 layer, d 1024, E 128; tiled -> this kernel):
// T 128 34 -> 17 us, T 512 34 -> 19 us, T 1024 34 -> 26 us; T 2048 keeps the tiled kernel
// (33 us against 42 with two tokens per warp).  PR-MoE E 64 (d 2048): T 256 60 -> 26 us,
// T 2048 61 -> 44 us.
int small_tokens_per_warp(int T, int E) {
  const long long etiles = (E + kSExp - 1) / kSExp, sms = sm_count();
  if (T <= 64 || etiles * ((T + kSWarps - 1) / kSWarps) <= sms) return 1;
  if (etiles * ((T + 2 * kSWarps - 1) / (2 * kSWarps)) <= 2 * sms) return 2;
  return 0;
}

template <typename Tin>
cudaError_t launch_small(const Tin* x, const float* Wg, int T, int d, int E, float* logits,
                         int m, cudaStream_t s) {
  auto go = [&](auto kern, int M, size_t smem) -> cudaError_t {
    const dim3 g((E + kSExp - 1) / kSExp, (T + kSWarps * M - 1) / (kSWarps * M));
    return launch_k(kern, g, 256, smem, s, false, x, Wg, T, d, E, logits);
  };
  if constexpr (sizeof(Tin) == 2) {  // 48 KB ring; fp32 rows would need more than the default
    if (m == 4)
      return go(gate_logits_small_kernel<Tin, 4>, 4, kSStages * small_slot_bytes<Tin, 4>());
  }
  if (m >= 2) return go(gate_logits_small_kernel<Tin, 2>, 2, kSStages * small_slot_bytes<Tin, 2>());
  return go(gate_logits_small_kernel<Tin, 1>, 1, kSStages * small_slot_bytes<Tin, 1>());
}

// ---------------------------------------------------------------------------------------
// Large batches: one warp per block computes a tile of 32 tokens x 64 experts, 8 x 8 outputs
// per thread (tokens 4g..4g+3 and 16+4g..16+4g+3 of the tile, experts 4h..4h+3 and
// 32+4h..32+4h+3), so each step of i takes four conflict-free 16-byte shared loads for 64
// multiply-adds.  Wg and token chunks of 32 columns stream through a two-deep cp.async ring;
// each chunk of token rows is widened to fp32 once (exact) into an i-major tile.  Every
// output's chain runs in one thread in ascending i, as in the kernels above.
constexpr int kWT = 32, kWE = 64, kWK = 32;

template <typename Tin>
struct WideSmem {
  static constexpr int kRowBytes = kWK * (int)sizeof(Tin) + 16;   // padded: conflict-free reads
  float ws[2][kWK][kWE];
  uint8_t xh[2][kWT * kRowBytes];
  float xs[kWK][kWT];
};

template <typename Tin>
__global__ void __launch_bounds__(32) gate_logits_wide_kernel(const Tin* __restrict__ x,
                                                              const float* __restrict__ Wg,
                                                              int T, int d, int E,
                                                              float* __restrict__ logits) {
  pdl_trigger();   // the top-k kernel may start its launch; it waits for these logits
  __shared__ __align__(16) WideSmem<Tin> sm;
  constexpr int kRow = WideSmem<Tin>::kRowBytes;
  constexpr int kPiece = 16 / (int)sizeof(Tin);                // values per 16-byte piece
  constexpr int kPieces = kWK / kPiece;                        // pieces per token row chunk
  const int lane = threadIdx.x;
  const int t0 = blockIdx.x * kWT, e0 = blockIdx.y * kWE;
  const int g = lane >> 3, h = lane & 7;
  const int nch = d / kWK;
  auto issue = [&](int c, int st) {
    const int k0 = c * kWK;
#pragma unroll
    for (int q = 0; q < kWK * kWE / 4 / 32; ++q) {             // Wg: 512 pieces
      const int idx = q * 32 + lane, row = idx >> 4, col = (idx & 15) * 4;
      cp_async16(&sm.ws[st][row][col], Wg + (size_t)(k0 + row) * E + e0 + col, 16);
    }
#pragma unroll
    for (int q = 0; q < kWT * kPieces / 32; ++q) {             // token rows
      const int idx = q * 32 + lane, tt = idx / kPieces, pc = idx % kPieces;
      const int t = t0 + tt;
      cp_async16(sm.xh[st] + tt * kRow + pc * 16, x + (size_t)min(t, T - 1) * d + k0 + pc * kPiece,
                 t < T ? 16 : 0);
    }
    cp_async_commit();
  };
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
  issue(0, 0);
  for (int c = 0; c < nch; ++c) {
    const int st = c & 1;
    if (c + 1 < nch) {
      issue(c + 1, st ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    {   // widen this lane's token row of the chunk into the i-major tile
      const uint8_t* row = sm.xh[st] + lane * kRow;
#pragma unroll
      for (int pc = 0; pc < kPieces; ++pc) {
        float f[kPiece];
        unpack16(*reinterpret_cast<const uint4*>(row + pc * 16), f, static_cast<const Tin*>(nullptr));
#pragma unroll
        for (int v = 0; v < kPiece; ++v) sm.xs[pc * kPiece + v][lane] = f[v];
      }
    }
    __syncwarp();
#pragma unroll 4
    for (int kk = 0; kk < kWK; ++kk) {                         // ascending i
      const float4 xa = *reinterpret_cast<const float4*>(&sm.xs[kk][4 * g]);
      const float4 xb = *reinterpret_cast<const float4*>(&sm.xs[kk][16 + 4 * g]);
      const float4 wa = *reinterpret_cast<const float4*>(&sm.ws[st][kk][4 * h]);
      const float4 wb = *reinterpret_cast<const float4*>(&sm.ws[st][kk][32 + 4 * h]);
      const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = __fmaf_rn(xv[i], wv[j], acc[i][j]);
    }
    __syncwarp();                                              // chunk st may be refilled
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + (i < 4 ? 4 * g + i : 16 + 4 * g + (i - 4));
    if (t >= T) continue;
    float* row = logits + (size_t)t * E + e0;
    *reinterpret_cast<float4*>(row + 4 * h) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    *reinterpret_cast<float4*>(row + 32 + 4 * h) =
        make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
}

struct PlainLoad {
  __device__ __forceinline__ float operator()(const float* p) const { return *p; }
};

// One warp per token: softmax over E (fp32) and top-k on the logits.
__global__ void __launch_bounds__(256) softmax_topk_kernel(const float* __restrict__ logits, int T,
                                                           int E, int k,
                                                           float* __restrict__ probs_out,
                                                           int32_t* __restrict__ topk_idx,
                                                           float* __restrict__ topk_w,
                                                           float* __restrict__ logits_copy) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const TopK r = softmax_topk_warp(logits + (size_t)t * E, E, k, lane, PlainLoad(),
                                   probs_out ? probs_out + (size_t)t * E : nullptr,
                                   logits_copy ? logits_copy + (size_t)t * E : nullptr);
  if (lane == 0) {
    for (int j = 0; j < k; ++j) {
      topk_idx[(size_t)t * k + j] = r.idx[j];
      topk_w[(size_t)t * k + j] = r.w[j];
    }
  }
}

}  // namespace

cudaError_t launch_gate_logits(const void* x, int dtype_f16, const float* Wg, int T, int d, int E,
                               float* logits, cudaStream_t s) {
  const bool aligned = (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                       (reinterpret_cast<uintptr_t>(Wg) & 15) == 0;
  const int m = small_tokens_per_warp(T, E);
  if (m > 0 && d % kSKC == 0 && E % 4 == 0 && aligned) {
    if (dtype_f16)
      MOE_LAUNCH(launch_small(static_cast<const __half*>(x), Wg, T, d, E, logits, m, s));
    else
      MOE_LAUNCH(launch_small(static_cast<const float*>(x), Wg, T, d, E, logits, m, s));
    return cudaGetLastError();
  }
  // The one-warp 32 x 64 tiles need several warps per SM to hide their latencies: they win
  // from about four tiles per SM (2.4B+MoE-128 layer, T = 16384: 444 -> 360 us) and lose with
  // fewer (350M+MoE-128, T = 4096, two tiles per SM: 44 -> 67 us).
  const long long wide_tiles = (long long)((T + kWT - 1) / kWT) * (E / kWE);
  const bool wide_ok = E % kWE == 0 && d % kWK == 0 && aligned &&
                       (reinterpret_cast<uintptr_t>(logits) & 15) == 0 &&
                       wide_tiles >= 4LL * sm_count();
  if (wide_ok) {
    const dim3 wg((T + kWT - 1) / kWT, E / kWE);
    if (dtype_f16)
      MOE_LAUNCH(launch_k(gate_logits_wide_kernel<__half>, wg, 32, 0, s, false,
                          static_cast<const __half*>(x), Wg, T, d, E, logits));
    else
      MOE_LAUNCH(launch_k(gate_logits_wide_kernel<float>, wg, 32, 0, s, false,
                          static_cast<const float*>(x), Wg, T, d, E, logits));
    return cudaGetLastError();
  }
  dim3 grid((T + kTT - 1) / kTT, (E + kTE - 1) / kTE);
  const bool vec = d % 8 == 0 && E % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(Wg) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
  const int vt = vec_tile_tokens(T, E);
  const dim3 vgrid((T + vt - 1) / vt, (E + kTE - 1) / kTE);
  if (dtype_f16) {
    const __half* xh = static_cast<const __half*>(x);
    if (vec) {
      if (vt == 64)
        MOE_LAUNCH(launch_k(gate_logits_kernel<__half, 64>, vgrid, 256, 0, s, false, xh, Wg, T, d,
                            E, logits));
      else if (vt == 32)
        MOE_LAUNCH(launch_k(gate_logits_kernel<__half, 32>, vgrid, 128, 0, s, false, xh, Wg, T, d,
                            E, logits));
      else
        MOE_LAUNCH(launch_k(gate_logits_kernel<__half, 16>, vgrid, 64, 0, s, false, xh, Wg, T, d,
                            E, logits));
    }
    else MOE_LAUNCH(launch_k(gate_logits_scalar_kernel<__half>, grid, 256, 0, s, false, xh, Wg, T,
                             d, E, logits));
  } else {
    const float* xf = static_cast<const float*>(x);
    if (vec) {
      if (vt == 64)
        MOE_LAUNCH(launch_k(gate_logits_kernel<float, 64>, vgrid, 256, 0, s, false, xf, Wg, T, d,
                            E, logits));
      else if (vt == 32)
        MOE_LAUNCH(launch_k(gate_logits_kernel<float, 32>, vgrid, 128, 0, s, false, xf, Wg, T, d,
                            E, logits));
      else
        MOE_LAUNCH(launch_k(gate_logits_kernel<float, 16>, vgrid, 64, 0, s, false, xf, Wg, T, d,
                            E, logits));
    }
    else MOE_LAUNCH(launch_k(gate_logits_scalar_kernel<float>, grid, 256, 0, s, false, xf, Wg, T, d,
                             E, logits));
  }
  return cudaGetLastError();
}

cudaError_t launch_softmax_topk(const float* logits, int T, int E, int k, float* probs_out,
                                int32_t* topk_idx, float* topk_w, float* logits_copy,
                                cudaStream_t s, bool pdl) {
  const int warps = 8;
  return launch_k(softmax_topk_kernel, (T + warps - 1) / warps, warps * 32, 0, s, pdl, logits, T, E,
                  k, probs_out, topk_idx, topk_w, logits_copy);
}

}  // namespace moe
