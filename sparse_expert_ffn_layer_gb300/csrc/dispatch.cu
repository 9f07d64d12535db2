// Capacity-limited dispatch: per-expert counts, exclusive scan, slot assignment in token
// order, overflow dropped.
//
// Reading (the pages define no per-expert token capacity; the "expert capacity" of the
// DeepSpeed-MoE review, "Phenomenon2", counts experts per token): capacity-factor rule
// C = ceil(cf T / E) per expert; the assignments
// (t, j) are taken token-major; an assignment's rank is the number of earlier assignments
// to the same expert; it is kept iff rank < C; expert e owns the compact slot range
// offsets[e] .. offsets[e] + kept[e] - 1 in token order.
//
// One block of 32 warps, no atomics.  Warp w owns a contiguous run of the assignment list.
// Pass 1: each warp walks its run 32 assignments at a time; lanes with equal experts are
// grouped by ballots over the bits of the expert index, so the rank inside the warp's run is the warp's running
// count for that expert (in shared memory, private to the warp) plus the number of
// lower lanes in the group.  Pass 2: per expert, an exclusive scan of the 32 warp counts
// gives each warp's base; kept = min(count, C); a block scan of kept gives the offsets.
// Pass 3: each assignment's global rank is base + local rank, which decides kept / dropped
// and the slot; perm and the slot weights are assembled in shared memory and written out
// coalesced.
//
// Token-sharded batches (counts_all != null): this call holds one shard of a batch split
// over ranks in token order, and counts_all [n_ranks, E] holds every shard's raw counts.
// The assignments of earlier shards come first in the batch's token order, so expert e's
// capacity left for this shard is max(0, C - sum over earlier shards of their counts), and
// the kept / dropped decisions equal those of the whole batch dispatched at once.
#include <algorithm>

#include "launch.h"

namespace moe {
namespace {

constexpr int kWarps = 32;
constexpr int kUnroll = 8;      // batches of 32 assignments whose loads are issued together
constexpr int kRegBatches = 8;  // runs of up to 8 x 32 assignments per warp stay in registers

// Lanes holding the same expert as this lane (valid lanes only; an invalid lane is alone):
// one ballot per bit of the expert index, which keeps lanes whose bit agrees.
__device__ __forceinline__ unsigned match_lanes(int e, bool valid, int nbits, int lane) {
  unsigned m = __ballot_sync(0xffffffffu, valid);
  for (int b = 0; b < nbits; ++b) {
    const bool bit = (e >> b) & 1;
    const unsigned set = __ballot_sync(0xffffffffu, bit && valid);
    m &= bit ? set : ~set;
  }
  return valid ? m : (1u << lane);
}

// kReg > 0: each warp's run (<= 32 kReg assignments) is loaded once and its experts, local
// ranks and gate weights stay in registers from pass 1 to pass 3.  kReg == 0: any length;
// local ranks go through slot_of.
template <int kReg>
__global__ void __launch_bounds__(1024) dispatch_kernel(
    const int32_t* __restrict__ topk_idx, int n, int k, int E, int C,
    int32_t* __restrict__ counts_raw, int32_t* __restrict__ kept, int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm, int32_t* __restrict__ slot_of, const float* __restrict__ topk_w,
    float* __restrict__ slot_w, int S_cap, int stage_out, const int32_t* __restrict__ counts_all,
    int rank) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                       // [kWarps][E]: running count, then warp base
  int32_t* offs = sm + kWarps * E;         // [E + 1]
  int32_t* wsum = offs + E + 1;            // [kWarps] scan scratch
  int32_t* capv = wsum + kWarps;           // [E] capacity left for this call, per expert
  int32_t* perm_s = capv + E;              // [S_cap] when stage_out: perm, written out coalesced
  float* slotw_s = reinterpret_cast<float*>(perm_s + S_cap);   // [S_cap] gate weight per slot
  const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int q = threadIdx.x; q < kWarps * E; q += blockDim.x) cnt[q] = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  const int L = (n + kWarps - 1) / kWarps;
  const int a_begin = min(n, w * L), a_end = min(n, a_begin + L);
  const unsigned lt_mask = (1u << lane) - 1u;

  // pass 1: rank inside the warp's run
  int ev_r[kReg > 0 ? kReg : 1], rv_r[kReg > 0 ? kReg : 1];
  float wv_r[kReg > 0 ? kReg : 1];
  if (kReg > 0) {
#pragma unroll
    for (int u = 0; u < kReg; ++u) {                     // one burst of loads for the whole run
      const int a = a_begin + 32 * u + lane;
      ev_r[u] = a < a_end ? topk_idx[a] : -1;
      wv_r[u] = (a < a_end && slot_w) ? topk_w[a] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kReg; ++u) {
      rv_r[u] = 0;
      if (a_begin + 32 * u >= a_end) continue;           // warp-uniform
      const int a = a_begin + 32 * u + lane;
      const int e = ev_r[u];
      const bool valid = a < a_end && (unsigned)e < (unsigned)E;   // out-of-range: dropped
      const unsigned grp = match_lanes(e, valid, nbits, lane);
      const int leader = __ffs(grp) - 1;
      int before = 0;
      if (valid) before = cnt[w * E + e];
      __syncwarp();
      if (valid) {
        rv_r[u] = before + __popc(grp & lt_mask);
        if (lane == leader) cnt[w * E + e] = before + __popc(grp);
      }
      __syncwarp();
    }
  } else {
    // local ranks are kept temporarily in slot_of; eight batches of loads in flight
    for (int base = a_begin; base < a_end; base += 32 * kUnroll) {
      int ev[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int a = base + 32 * u + lane;
        ev[u] = a < a_end ? topk_idx[a] : -1;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (base + 32 * u >= a_end) break;               // warp-uniform
        const int a = base + 32 * u + lane;
        const int e = ev[u];
        const bool valid = a < a_end && (unsigned)e < (unsigned)E;
        const unsigned grp = match_lanes(e, valid, nbits, lane);
        const int leader = __ffs(grp) - 1;
        int before = 0;
        if (valid) before = cnt[w * E + e];
        __syncwarp();
        if (valid) {
          slot_of[a] = before + __popc(grp & lt_mask);
          if (lane == leader) cnt[w * E + e] = before + __popc(grp);
        }
        __syncwarp();
      }
    }
  }
  __syncthreads();

  // pass 2: per-expert scan over warps, kept, then a block scan of kept
  int my_kept = 0;
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int run = 0;
    for (int ww = 0; ww < kWarps; ++ww) {
      int c = cnt[ww * E + e];
      cnt[ww * E + e] = run;
      run += c;
    }
    counts_raw[e] = run;
    int cap = C;
    if (counts_all) {
      int before = 0;                                   // earlier shards' assignments to e
      for (int r = 0; r < rank; ++r) before += counts_all[(size_t)r * E + e];
      cap = max(0, C - before);
    }
    capv[e] = cap;
    my_kept = min(run, cap);
    kept[e] = my_kept;
  }
  // block-wide exclusive scan of my_kept over threads 0 .. E-1 (E <= 1024)
  int incl = my_kept;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    int v = wsum[lane];
    int s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    wsum[lane] = s - v;                  // exclusive prefix of warp totals
  }
  __syncthreads();
  if (threadIdx.x < E) {
    int ex = wsum[w] + incl - my_kept;
    offs[threadIdx.x] = ex;
    offsets[threadIdx.x] = ex;
    if (threadIdx.x == E - 1) {
      offs[E] = ex + my_kept;
      offsets[E] = ex + my_kept;
    }
  }
  __syncthreads();

  // pass 3: global rank -> slot
  auto place = [&](int a, int e, int rank_local, float wgt) {
    if ((unsigned)e >= (unsigned)E) {
      slot_of[a] = -1;
      return;
    }
    const int r = cnt[w * E + e] + rank_local;
    if (r < capv[e]) {
      const int s = offs[e] + r;
      slot_of[a] = s;
      if (stage_out) {
        perm_s[s] = a / k;
        if (slot_w) slotw_s[s] = wgt;
      } else {
        perm[s] = a / k;
        if (slot_w) slot_w[s] = wgt;
      }
    } else {
      slot_of[a] = -1;
    }
  };
  if (kReg > 0) {
#pragma unroll
    for (int u = 0; u < kReg; ++u) {
      const int a = a_begin + 32 * u + lane;
      if (a < a_end) place(a, ev_r[u], rv_r[u], wv_r[u]);
    }
  } else {
    for (int base = a_begin; base < a_end; base += 32 * kUnroll) {
      int ev[kUnroll], rv[kUnroll];
      float wv[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int a = base + 32 * u + lane;
        ev[u] = a < a_end ? topk_idx[a] : -1;
        rv[u] = a < a_end ? slot_of[a] : 0;
        wv[u] = (a < a_end && slot_w) ? topk_w[a] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int a = base + 32 * u + lane;
        if (a < a_end) place(a, ev[u], rv[u], wv[u]);
      }
    }
  }
  if (stage_out) {                                       // coalesced copy-out of the slots
    __syncthreads();
    const int S = offs[E];
    for (int q = threadIdx.x; q < S; q += blockDim.x) perm[q] = perm_s[q];
    if (slot_w)
      for (int q = threadIdx.x; q < S; q += blockDim.x) slot_w[q] = slotw_s[q];
  }
}

}  // namespace

size_t dispatch_smem_bytes(int E) {
  return sizeof(int32_t) * ((size_t)kWarps * E + E + 1 + kWarps + E);
}

// Slots staged in shared memory when they fit beside the counters.
constexpr size_t kDispatchSmemMax = 200 * 1024;

cudaError_t launch_dispatch(const int32_t* topk_idx, int T, int k, int E, int C, int32_t* counts_raw,
                            int32_t* kept, int32_t* offsets, int32_t* perm, int32_t* slot_of,
                            const float* topk_w, float* slot_w, cudaStream_t s, bool pdl,
                            const int32_t* counts_all, int rank) {
  const int n = T * k;
  const int S_cap = (int)std::min<long long>(n, (long long)E * C);
  size_t smem = dispatch_smem_bytes(E);
  const size_t staged = smem + (size_t)S_cap * 8;
  const int stage_out = staged <= kDispatchSmemMax ? 1 : 0;
  if (stage_out) smem = staged;
  const bool in_regs = (n + kWarps - 1) / kWarps <= 32 * kRegBatches;
  auto kern = in_regs ? dispatch_kernel<kRegBatches> : dispatch_kernel<0>;
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(kern));
  if (err != cudaSuccess) return err;
  return launch_k(kern, 1, kWarps * 32, smem, s, pdl, topk_idx, n, k, E, C, counts_raw, kept,
                  offsets, perm, slot_of, topk_w, slot_w, S_cap, stage_out, counts_all, rank);
}

}  // namespace moe
