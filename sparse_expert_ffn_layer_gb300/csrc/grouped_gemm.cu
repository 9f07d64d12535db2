// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// Both GEMMs of the expert FFN run "swap-AB": the weight tile is the MMA's M = 128 operand
// (A, read M-major straight from the row-major weights) and the tokens are the N operand
// (B, K-major rows), so N is the ragged per-expert row count, rounded up to 16.
//
//   GEMM1  H[s, :]   = GeLU_tanh(X[perm[s], :] . W1[e])     A = W1[e]^T tile, B = gathered X rows
//   GEMM2  out[t, :] (+)= w_s (H[s, :] . W2[e])              A = W2[e]^T tile, B = H rows
//
// Weight streaming dominates the bytes of the layer at every configured size: reading the
// expert weights from memory is the bottleneck of MoE inference (DeepSpeed-MoE review,
// "PR-MoE and MoS"), and small-batch GEMMs are bound by memory bandwidth (DeepSpeed
// Inference review, "제안 방법").  So each (expert, M-tile) weight tile is read once, by one
// CTA, through a deep TMA pipeline, while the token rows come from L2.
//
// Kernel shape: persistent, one CTA per SM.
//   warp 0      producer: TMA of the A tile (two 64-wide boxes, 128-byte swizzle) and of the
//               B rows (tile::gather4 through perm, or 16-row boxes of contiguous rows)
//   warp 1      TMEM allocation and the MMA issue (one elected lane)
//   warps 2..   epilogue (eight warps, four in the decode-sized variant): tcgen05.ld of the
//               fp32 accumulator, GeLU / gate-weighted combine, stores; TMEM accumulators in a
//               ring of slots so the epilogue of one item overlaps the next item's MMAs.
// Work items are (tile of <= nmax rows of one group, M-tile), groups being the experts in
// slot order plus, for the residual variant, one group of all T tokens using the dense MLP
// weights (PR-MoE's fixed MLP, DeepSpeed-MoE review "Phenomenon2": Residual-MoE).
// Every wait is bounded: a stalled pipeline records MOE_ERR_TIMEOUT and the CTA leaves.
#include <algorithm>

#include "launch.h"

namespace moe {
namespace {

// Warps: producer, MMA, then the epilogue warps: eight (two per TMEM lane quarter, taking
// alternate 16-column chunks) for full-size items, so that an item's accumulator slots drain
// in half the time and the next item's MMAs wait less (with 160-row tiles only three slots
// fit TMEM; first GEMM of the 2.4B top-2 layer at T = 16384: 2390 -> 2327 us with eight
// instead of four); four for the decode-sized variant, whose items are a few columns wide.
template <bool kSplit>
struct Roles {
  static constexpr int kEpiWarps = kSplit ? 4 : 8;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
};
constexpr int kBM = 128;          // MMA M (weight rows per accumulator)
constexpr int kBK = 64;           // K per pipeline stage (one 128-byte swizzle span of f16)
constexpr int kABytes = kBM * kBK * 2;   // one 128-row A block per stage; an item has mw of them
constexpr int kMaxSlots = 16;     // TMEM accumulator slots (512 columns / at least 32 each)

struct SmemLayout {
  uint32_t stage_bytes, b_off, bars_off, misc_off, rows_off, total;
};

__host__ __device__ inline SmemLayout smem_layout(int nmax, int stages, int E, int mw,
                                                  int epi_warps) {
  SmemLayout L;
  L.b_off = (uint32_t)mw * kABytes;
  L.stage_bytes = L.b_off + (uint32_t)nmax * 128u;
  uint32_t off = (uint32_t)stages * L.stage_bytes;
  L.bars_off = off;
  off += (uint32_t)(2 * stages + 2 * kMaxSlots) * 8u;
  L.misc_off = off;
  off += 16u + 8u * (uint32_t)(E + 1);       // tmem base, abort flag, chunk prefix, offsets
  L.rows_off = off;
  off += (uint32_t)epi_warps * 2u * 4u * (uint32_t)nmax;  // per epilogue warp [nmax] tokens
                                                          // and gate weights
  L.total = off + 1024u;                     // slack for 1024-byte alignment
  return L;
}

struct Tile {
  int res;      // 1: residual group
  int e;        // expert (res == 0)
  int row0;     // first row of the tile: slot (experts) or token (residual)
  int n;        // valid rows
  int mt;       // M-tile index
  int K;        // shared dimension
};

// Maps work item i to its tile.  prefix[e] = chunks of experts < e (prefix[E] = total).
__device__ __forceinline__ Tile decode(int i, const GemmArgs& a, const int32_t* prefix,
                                       const int32_t* offs) {
  // Items of one group are ordered weight block major, row tile minor, so the row tiles that
  // read the same weight block run side by side on neighbouring CTAs and share it in L2.
  Tile t;
  const int n_exp = prefix[a.E] * a.mt_exp;
  if (i < n_exp) {
    int lo = 0, hi = a.E;                   // largest e with prefix[e] * mt_exp <= i
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (prefix[mid] * a.mt_exp <= i) lo = mid; else hi = mid;
    }
    const int chunks = prefix[lo + 1] - prefix[lo];
    const int local = i - prefix[lo] * a.mt_exp;
    t.mt = local / chunks;
    const int chunk = local - t.mt * chunks;
    t.res = 0;
    t.e = lo;
    const int kept = max(0, offs[lo + 1] - offs[lo]);
    t.row0 = offs[lo] + chunk * a.nmax;
    t.n = min(a.nmax, kept - chunk * a.nmax);
    t.K = a.K;
  } else {
    const int chunks = (a.n_res_rows + a.nmax - 1) / a.nmax;
    const int local = i - n_exp;
    t.mt = local / chunks;
    const int chunk = local - t.mt * chunks;
    t.res = 1;
    t.e = 0;
    t.row0 = chunk * a.nmax;
    t.n = min(a.nmax, a.n_res_rows - t.row0);
    t.K = a.K_res;
  }
  return t;
}

// kSplit: the decode-sized variant, whose items are cut into K chunks (fp32 partial sums,
// summed by a reduce kernel); a template parameter so that neither variant carries the other's
// epilogue code (at decode sizes the kernel's fixed costs decide its time).
template <bool kGatherB, int kEpi, int kMW, bool kSplit>
__global__ void __launch_bounds__(Roles<kSplit>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmA_res,
                        const __grid_constant__ CUtensorMap tmB_res, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int kEpiWarps = Roles<kSplit>::kEpiWarps;
  constexpr int kEpiThreads = 32 * kEpiWarps;
  const SmemLayout L = smem_layout(a.nmax, a.stages, a.E, a.mw, kEpiWarps);
  constexpr int mw = kMW;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars_off);
  uint64_t* empty = full + a.stages;
  // TMEM accumulators form a ring of nslots slots of acc_cols columns.  Item j (the j-th
  // item of this CTA) accumulates its mw weight blocks in slots (j mw + h) mod nslots; the
  // MMA warp waits for the item's slots to be drained (acc_empty[slot]) before its first MMA,
  // and the epilogue releases each slot as soon as it has read it, so the next item's MMAs
  // overlap the epilogue whenever nslots >= 2 mw (partly when nslots > mw).
  // acc_full[j mod nslots] completes when item j's MMAs are done.
  uint64_t* acc_full = empty + a.stages;     // [nslots]
  uint64_t* acc_empty = acc_full + kMaxSlots;  // [nslots]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + L.misc_off + 16);
  int32_t* soffs = prefix + (a.E + 1);                     // copy of offsets[0 .. E]
  int32_t* row_tok = reinterpret_cast<int32_t*>(smem + L.rows_off);   // [epilogue warps][nmax]
  float* row_w = reinterpret_cast<float*>(row_tok + kEpiWarps * a.nmax);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < a.nslots; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiThreads);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (a.n_res_rows > 0) {
      prefetch_tmap(&tmA_res);
      prefetch_tmap(&tmB_res);
    }
  }
  if (warp == 1) tmem_alloc(tmem_holder, a.tmem_cols);
  // Everything above is independent of the previous kernel of the stream.  With early_a the
  // routing (offsets) comes from a kernel at least two launches back, which has completed by
  // the time this grid starts (every kernel of the chain waits for its predecessor before it
  // lets its successor launch), and the weights are never written: so the item list is built
  // and the producer issues the weight loads of its first stages before the wait.
  if (!a.early_a) {
    pdl_wait();
    pdl_trigger();
  }
  // chunk prefix over experts (warp 2), E <= 1024
  if (warp == 2) {
    // offsets clamped to [0, S_bound]: offsets[E] beyond the caller's S_max cannot make a
    // tile write past H or the output, and decreasing offsets give empty groups (kept is
    // taken as max(0, .) below); either records MOE_ERR_DEVICE_BOUNDS
    bool bad = false;
    for (int e = lane; e <= a.E; e += 32) {
      const int o = __ldcg(a.offsets + e);
      soffs[e] = min(max(o, 0), a.S_bound);
      bad |= soffs[e] != o;
    }
    __syncwarp();
    for (int e = lane; e < a.E; e += 32) bad |= soffs[e + 1] < soffs[e];
    if (bad) record_status(a.status, kErrBounds);
    const int per = (a.E + 31) / 32;
    const int e_lo = lane * per, e_hi = min(a.E, e_lo + per);
    int local = 0;
    for (int e = e_lo; e < e_hi; ++e) {
      const int kept = max(0, soffs[e + 1] - soffs[e]);
      local += (kept + a.nmax - 1) / a.nmax;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int e = e_lo; e < e_hi; ++e) {
      prefix[e] = run;
      const int kept = max(0, soffs[e + 1] - soffs[e]);
      run += (kept + a.nmax - 1) / a.nmax;
    }
    if (lane == 31) prefix[a.E] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int n_exp_items = prefix[a.E] * a.mt_exp;
  const int n_res_items = a.n_res_rows > 0 ? ((a.n_res_rows + a.nmax - 1) / a.nmax) * a.mt_res : 0;
  const int ksplit = kSplit ? a.ksplit : 1;
  const int total = (n_exp_items + n_res_items) * ksplit;

  uint32_t issued = 0, issued_parity = 0;     // producer: stages with a fill in flight
  // early_a: weight loads of the first stages, issued before the wait (their stages' token
  // rows follow after it, in the main loop below)
  int n_early = 0;
  if (a.early_a && warp == 0 && lane == 0) {
    int stage = 0;
    for (int i = blockIdx.x; i < total && n_early < a.stages; i += gridDim.x) {
      const Tile t = decode(i / ksplit, a, prefix, soffs);
      const int ks = i - (i / ksplit) * ksplit;
      const int npad = max(16, (t.n + 15) & ~15);
      const CUtensorMap* mA = t.res ? &tmA_res : &tmA;
      const int a_y0 = t.res ? 0 : t.e * a.a_rows_per_expert;
      const int a_x = t.mt * mw * kBM;
      const int nkb = t.K / kBK;
      const int kb0 = ks * nkb / ksplit, kb1 = (ks + 1) * nkb / ksplit;
      for (int kb = kb0; kb < kb1 && n_early < a.stages; ++kb, ++n_early, ++stage) {
        uint8_t* sA = smem + (size_t)stage * L.stage_bytes;
        mbar_expect_tx(&full[stage], (uint32_t)(mw * kABytes) + (uint32_t)npad * 128u);
#pragma unroll
        for (int h = 0; h < mw; ++h) {
          tma_load_2d(sA + h * kABytes, mA, a_x + h * kBM, a_y0 + kb * kBK, &full[stage]);
          tma_load_2d(sA + h * kABytes + kABytes / 2, mA, a_x + h * kBM + 64, a_y0 + kb * kBK,
                      &full[stage]);
        }
        issued |= 1u << stage;                   // phase 0 of a fresh stage
      }
    }
  }
  if (a.early_a) {
    pdl_wait();
    pdl_trigger();
  }
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    n_early = __shfl_sync(0xffffffffu, n_early, 0);
    int it = 0;                                   // k-iterations so far (the first n_early
                                                  // have their weight loads in flight)
    bool bad_row = false;
    // this lane's gather rows (first GEMM): groups g = lane, lane + 32 of four rows each;
    // the next tile's rows are fetched while the current tile streams.  A perm entry outside
    // [0, T) is replaced by row 0 and reported once at the end.
    auto load_rows = [&](const Tile& t, int (&rows)[2][4]) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = 4 * (lane + 32 * h) + q;
          const int src = t.row0 + (r < t.n ? r : 0);
          const int tok = t.res ? src : a.perm[src];
          const bool oob = (unsigned)tok >= (unsigned)a.n_tokens;
          bad_row |= oob;
          rows[h][q] = oob ? 0 : tok;
        }
    };
    int rows[2][4], rows_next[2][4];
    if (kGatherB && blockIdx.x < total) load_rows(decode(blockIdx.x / ksplit, a, prefix, soffs), rows);
    for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x) {
      const Tile t = decode(i / ksplit, a, prefix, soffs);
      const int ks = i - (i / ksplit) * ksplit;
      const int npad = max(16, (t.n + 15) & ~15);
      const CUtensorMap* mA = t.res ? &tmA_res : &tmA;
      const CUtensorMap* mB = t.res ? &tmB_res : &tmB;
      const int a_y0 = t.res ? 0 : t.e * a.a_rows_per_expert;
      const int a_x = t.mt * mw * kBM;
      if (kGatherB && i + (int)gridDim.x < total)
        load_rows(decode((i + gridDim.x) / ksplit, a, prefix, soffs), rows_next);
      const int nkb = t.K / kBK;
      const int kb0 = ks * nkb / ksplit, kb1 = (ks + 1) * nkb / ksplit;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        uint8_t* sA = smem + (size_t)stage * L.stage_bytes;
        uint8_t* sB = sA + L.b_off;
        if (it >= n_early) {                          // else: weights already in flight
          bool ok = true;
          if (lane == 0) ok = mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status, a.wait_ns);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (lane == 0) {
            mbar_expect_tx(&full[stage], (uint32_t)(mw * kABytes) + (uint32_t)npad * 128u);
#pragma unroll
            for (int h = 0; h < mw; ++h) {               // mw adjacent 128-row blocks
              tma_load_2d(sA + h * kABytes, mA, a_x + h * kBM, a_y0 + kb * kBK, &full[stage]);
              tma_load_2d(sA + h * kABytes + kABytes / 2, mA, a_x + h * kBM + 64, a_y0 + kb * kBK,
                          &full[stage]);
            }
          }
          __syncwarp();
        }
        if (kGatherB) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int g = lane + 32 * h;
            if (4 * g < npad)
              tma_gather4(sB + g * 512, mB, kb * kBK, rows[h][0], rows[h][1], rows[h][2], rows[h][3],
                          &full[stage]);
          }
        } else {
          for (int b = lane; b < npad / 16; b += 32)
            tma_load_2d(sB + b * 2048, mB, kb * kBK, t.row0 + 16 * b, &full[stage]);
        }
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == a.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (kGatherB) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int q = 0; q < 4; ++q) rows[h][q] = rows_next[h][q];
      }
    }
    if (kGatherB && __any_sync(0xffffffffu, bad_row) && lane == 0) record_status(a.status, kErrBounds);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x, ++local) {
      const Tile t = decode(i / ksplit, a, prefix, soffs);
      const int ks = i - (i / ksplit) * ksplit;
      const int npad = max(16, (t.n + 15) & ~15);
      const uint32_t blk0 = (uint32_t)local * mw;        // ring position of block 0
      uint32_t d_tmem[mw];
#pragma unroll
      for (int h = 0; h < mw; ++h) d_tmem[h] = tmem_base + ((blk0 + h) % a.nslots) * a.acc_cols;
      // the item's accumulator slots must have been drained by the epilogue
      bool ok = true;
      if (lane == 0) {
        for (int h = 0; h < mw && ok; ++h) {
          const uint32_t blk = blk0 + h;
          ok = mbar_wait_bounded(&acc_empty[blk % a.nslots], ((blk / a.nslots) & 1u) ^ 1u,
                                 abort_flag, a.status, a.wait_ns);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const uint32_t idesc = idesc_f16(kBM, npad, 1, 0);
      const int nkb = t.K / kBK;
      const int kb0 = ks * nkb / ksplit, kb1 = (ks + 1) * nkb / ksplit;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (lane == 0) ok = mbar_wait_bounded(&full[stage], phase, abort_flag, a.status, a.wait_ns);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(smem + (size_t)stage * L.stage_bytes);
          // descriptors of the stage's first A block and B rows; the others differ only in
          // the start address (in 16-byte units, bits 0..13, which shared-memory addresses
          // below 256 KB never carry out of)
          const uint64_t ad0 = smem_desc(a0, a.a_lbo, a.a_sbo, 2);
          const uint64_t bd0 = smem_desc(a0 + L.b_off, 16, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t bd = bd0 + (uint64_t)(kk * 32 / 16);
#pragma unroll
            for (int h = 0; h < mw; ++h) {             // same token rows, mw weight blocks
              const uint64_t ad = ad0 + (uint64_t)((h * kABytes + kk * 2048) / 16);
              tc_mma_f16(d_tmem[h], ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
            }
          }
          tc_commit(&empty[stage]);        // frees the stage once these MMAs have read it
        }
        __syncwarp();
        if (++stage == a.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&acc_full[local % a.nslots]);
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..)
    const int quarter = warp & 3;                  // TMEM lanes 32*quarter .. +31
    const int half = (warp - 2) >> 2;              // which 16-column chunks: c0 / 16 = half mod
    const int row_in_tile = 32 * quarter + lane;   // (epilogue warps / 4)
    if (kEpi == kEpiGeluH) {
      // pre-work while the first tiles stream in: zero buffers the next kernel accumulates into
      const int ep_tid = blockIdx.x * kEpiThreads + (threadIdx.x - 64);
      const int ep_threads = gridDim.x * kEpiThreads;
      if (a.zero_buf) {
        uint4* z4 = reinterpret_cast<uint4*>(a.zero_buf);
        const size_t n4 = a.zero_bytes / 16;
        for (size_t q = ep_tid; q < n4; q += ep_threads) z4[q] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (a.drop_out) {
        const int gw = ep_tid >> 5, nw = ep_threads >> 5;
        for (int tok = gw; tok < a.drop_T; tok += nw) {
          if (a.drop_slot_of[tok] >= 0) continue;
          uint4* row = reinterpret_cast<uint4*>(a.drop_out + (size_t)tok * a.drop_d);
          for (int c = lane; c < a.drop_d / 8; c += 32) row[c] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    int local = 0;
    for (int i = blockIdx.x; i < total && !*abort_flag; i += gridDim.x, ++local) {
      const Tile t = decode(i / ksplit, a, prefix, soffs);
      const int ks = i - (i / ksplit) * ksplit;
      // second GEMM: each warp stages the tile's tokens and gate weights in its own shared
      // memory while the accumulator is still being computed (a load per row per warp
      // instead of one per row per thread; warp-private, so no cross-warp barrier)
      const bool scatter = kEpi == kEpiCombine && !t.res && a.mode != kModeExpertOut && !kSplit;
      int32_t* rt = row_tok + (warp - 2) * a.nmax;
      float* rw = row_w + (warp - 2) * a.nmax;
      if (scatter) {
        for (int r = lane; r < t.n; r += 32) {
          rt[r] = a.perm[t.row0 + r];
          rw[r] = a.slot_w[t.row0 + r];
        }
      }
      __syncwarp();
      bool ok = true;
      if (lane == 0)
        ok = mbar_wait_bounded(&acc_full[local % a.nslots], (uint32_t)(local / a.nslots) & 1u,
                               abort_flag, a.status, a.wait_ns);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int h = 0; h < mw; ++h) {
      const int m = (t.mt * mw + h) * kBM + row_in_tile;
      const uint32_t slot = ((uint32_t)local * mw + h) % a.nslots;
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + slot * a.acc_cols;
      for (int c0 = 16 * half; c0 < t.n; c0 += 16 * (kEpiWarps / 4)) {
        float v[16];
        tmem_ld16(taddr + (uint32_t)c0, v);
        if (kEpi == kEpiGeluH && !kSplit) {
          // GeLU -> f16 H, two columns per 4-byte store: lanes 2i and 2i+1 hold columns m and
          // m+1; for each pair of tokens the even lane stores token 2p of both columns and the
          // odd lane token 2p+1, each taking the neighbour's value by one shuffle
          __half* hbase = t.res ? a.hres_out : a.h_out;
          const size_t ld = t.res ? (size_t)a.ldhres : (size_t)a.ldh;
          const bool odd = lane & 1;
#pragma unroll
          for (int p2 = 0; p2 < 8; ++p2) {
            const float g0 = gelu_tanh(v[2 * p2]), g1 = gelu_tanh(v[2 * p2 + 1]);
            const float recv = __shfl_xor_sync(0xffffffffu, odd ? g0 : g1, 1);
            const int s = c0 + 2 * p2 + (odd ? 1 : 0);
            if (s < t.n)
              *reinterpret_cast<__half2*>(hbase + (size_t)(t.row0 + s) * ld + (m & ~1)) =
                  odd ? __floats2half2_rn(recv, g1) : __floats2half2_rn(g0, recv);
          }
          continue;
        }
        if (kEpi == kEpiCombine && !kSplit && a.mode == kModeSum) {
          // out += f16(w * acc), two columns per f16x2 reduction (lanes 2i, 2i+1 hold columns
          // m, m+1; the even lane takes token 2p of both, the odd lane token 2p+1); residual
          // rows are token rows with weight 1
#pragma unroll
          for (int p2 = 0; p2 < 8; ++p2) {
            const bool odd = lane & 1;
            const float recv = __shfl_xor_sync(0xffffffffu, odd ? v[2 * p2] : v[2 * p2 + 1], 1);
            const int s = c0 + 2 * p2 + (odd ? 1 : 0);
            if (s < t.n) {
              const int tok = t.res ? t.row0 + s : rt[s];
              const float w = t.res ? 1.0f : rw[s];
              const float lo = odd ? recv : v[2 * p2], hi = odd ? v[2 * p2 + 1] : recv;
              red_add_f16x2(a.out + (size_t)tok * a.ldo + (m & ~1), __floats2half2_rn(w * lo, w * hi));
            }
          }
          continue;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int s = c0 + j;
          if (s >= t.n) break;
          const int row = t.row0 + s;
          if (kSplit) {
            const int prow = t.res ? a.part_res_row0 + row : row;
            a.partial[((size_t)ks * a.part_rows + prow) * a.part_cols + m] = v[j];
          } else if (kEpi == kEpiGeluH) {
            // (handled above)
          } else {
            if (t.res) {
              a.r32[(size_t)row * a.ldo + m] = v[j];
            } else if (a.mode == kModeExpertOut) {
              a.out[(size_t)row * a.ldo + m] = __float2half_rn(v[j]);
            } else {
              const int tok = rt[s];
              const float w = rw[s];
              if (a.mode == kModeDirect) a.out[(size_t)tok * a.ldo + m] = __float2half_rn(w * v[j]);
              else red_add_f32(a.acc32 + (size_t)tok * a.ldo + m, w * v[j]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[slot]);       // this block's slot may take the next MMAs
      }
    }
  }

  // ------------------------------------------------------------ teardown
  if (*abort_flag && warp == 0 && lane == 0) {
    // let the last copy issued into each stage land before the CTA's shared memory is
    // released (bounded: 100 ms per stage)
    for (int s = 0; s < a.stages; ++s) {
      if (!(issued >> s & 1u)) continue;
      const uint32_t par = issued_parity >> s & 1u;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&full[s], par)) {
        if (globaltimer_ns() - t0 > 100000000ull) break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, a.tmem_cols);
}

// Dynamic shared memory of a launch is at least this much, so that no two CTAs of these
// kernels are ever resident on one SM (an SM has 228 KB): a CTA that starts early under
// programmatic dependent launch can then never wait in tcgen05.alloc for columns held by a
// CTA of the previous GEMM on the same SM.
constexpr size_t kMinGemmSmem = 116 * 1024;

template <bool G, int Epi, int MW, bool Split>
cudaError_t launch_mw(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Ar,
                      const CUtensorMap& Br, const GemmArgs& args, int grid, cudaStream_t s,
                      bool pdl) {
  const SmemLayout L = smem_layout(args.nmax, args.stages, args.E, MW, Roles<Split>::kEpiWarps);
  auto kern = grouped_gemm_kernel<G, Epi, MW, Split>;
  cudaError_t err = ensure_smem_attr(reinterpret_cast<const void*>(kern));
  if (err != cudaSuccess) return err;
  return launch_k(kern, grid, Roles<Split>::kThreads, std::max<size_t>(L.total, kMinGemmSmem), s,
                  pdl, A, B, Ar, Br, args);
}

template <bool G, int Epi, bool Split>
cudaError_t launch_split(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Ar,
                         const CUtensorMap& Br, const GemmArgs& args, int grid, cudaStream_t s,
                         bool pdl) {
  switch (args.mw) {
    case 1: return launch_mw<G, Epi, 1, Split>(A, B, Ar, Br, args, grid, s, pdl);
    case 2: return launch_mw<G, Epi, 2, Split>(A, B, Ar, Br, args, grid, s, pdl);
    case 4: return launch_mw<G, Epi, 4, Split>(A, B, Ar, Br, args, grid, s, pdl);
  }
  return cudaErrorInvalidValue;
}

template <bool G, int Epi>
cudaError_t launch_one(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Ar,
                       const CUtensorMap& Br, const GemmArgs& args, int grid, cudaStream_t s,
                       bool pdl) {
  return args.ksplit > 1 ? launch_split<G, Epi, true>(A, B, Ar, Br, args, grid, s, pdl)
                         : launch_split<G, Epi, false>(A, B, Ar, Br, args, grid, s, pdl);
}

}  // namespace

int gemm_stages_for(int nmax, int E, int mw, int smem_limit) {
  // the larger (full-size) epilogue's staging, so that the count holds for either variant
  for (int st = 8; st >= 2; --st)
    if ((int)smem_layout(nmax, st, E, mw, Roles<false>::kEpiWarps).total <= smem_limit) return st;
  return 0;
}

cudaError_t launch_grouped_gemm1(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Ar,
                                 const CUtensorMap& Br, const GemmArgs& args, int grid,
                                 cudaStream_t s, bool pdl) {
  return launch_one<true, kEpiGeluH>(A, B, Ar, Br, args, grid, s, pdl);
}

cudaError_t launch_grouped_gemm2(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Ar,
                                 const CUtensorMap& Br, const GemmArgs& args, int grid,
                                 cudaStream_t s, bool pdl) {
  return launch_one<false, kEpiCombine>(A, B, Ar, Br, args, grid, s, pdl);
}

cudaError_t launch_grouped_gemm1_rows(const CUtensorMap& A, const CUtensorMap& B,
                                      const CUtensorMap& Ar, const CUtensorMap& Br,
                                      const GemmArgs& args, int grid, cudaStream_t s, bool pdl) {
  return launch_one<false, kEpiGeluH>(A, B, Ar, Br, args, grid, s, pdl);
}

}  // namespace moe
