// C-ABI front end (include/moe.h): argument checks, workspace carving, TMA descriptors and the
// launch sequence of each entry point.  All device work is in the kernels of this library.
#include <math.h>
#include <cmath>
#include <cstdlib>
#include <mutex>
#include <set>
#include <utility>

#include "../../include/moe.h"
#include "launch.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxE = 1024;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int capacity_of(int T, int E, float cf) {
  if (T < 0 || E < 1 || !(cf > 0.0f)) return -1;
  if (T == 0) return 0;
  if (isinf(cf)) return T;              // dropless: no expert receives more than T assignments
  double c = ceil((double)cf * (double)T / (double)E);
  if (c > 2147483647.0) return -1;
  return (int)c;
}

// ---------------------------------------------------------------- workspace layout
// Token rows per tile of the first (gathering) GEMM.
constexpr int kGather1Rows = 64;

// Split-K applies to decode-sized batches only: at most kMaxSplit chunks, and only when the
// expert slots plus residual rows fit in kSplitRows (the fp32 partial sums then stay small).
constexpr int kMaxSplit = 32;
constexpr int kSplitRows = 64;

struct Ws {
  size_t status, logits, topk_idx, topk_w, counts, kept, offsets, perm, slot_w, slot_of, H, Hres,
      acc32, r32, partial, partial_bytes, Xg, total;
};

Ws ws_layout(int T, int d, int f, int E, int k, int C, bool residual, int f_res, bool f16) {
  const size_t elt = f16 ? 2 : 4;
  const size_t S_max = (size_t)std::min<long long>((long long)T * k, (long long)E * C);
  const bool accum = k == 2 && residual;     // three addends per output: fp32, fixed order
  Ws w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off += align_up(bytes);
    return at;
  };
  w.status = take(kAlign);
  w.H = take(std::max<size_t>(S_max, 1) * f * elt);
  w.logits = take((size_t)T * E * 4);
  w.topk_idx = take((size_t)T * k * 4);
  w.topk_w = take((size_t)T * k * 4);
  w.counts = take((size_t)E * 4);
  w.kept = take((size_t)E * 4);
  w.offsets = take((size_t)(E + 1) * 4);
  w.perm = take(std::max<size_t>(S_max, 1) * 4);
  w.slot_w = take(std::max<size_t>(S_max, 1) * 4);
  w.slot_of = take((size_t)T * k * 4);
  w.Hres = residual ? take((size_t)T * f_res * elt) : 0;
  w.acc32 = accum ? take((size_t)T * d * 4) : 0;
  w.r32 = residual ? take((size_t)T * d * 4) : 0;
  const size_t part_rows = S_max + (residual ? (size_t)T : 0);
  w.partial_bytes = 0;
  w.partial = 0;
  if (f16 && part_rows <= (size_t)kSplitRows) {
    const size_t cols = std::max<size_t>(std::max(f, d), residual ? f_res : 0);
    w.partial_bytes = (size_t)kMaxSplit * part_rows * cols * 4;
    w.partial = take(w.partial_bytes);
  }
  // slot-ordered copy of the kept token rows, for batches whose experts hold more rows than
  // one gathered tile (see run_tc_ffn)
  w.Xg = (f16 && std::min(C, T) > kGather1Rows) ? take(std::max<size_t>(S_max, 1) * d * elt) : 0;
  w.total = off;
  return w;
}

size_t expert_ffn_ws_bytes(int S_max, int f, bool f16) {
  return kAlign + align_up(std::max<size_t>((size_t)S_max, 1) * f * (f16 ? 2 : 4));
}

// ---------------------------------------------------------------- argument checks
moe_status check_shape(int T, int d, int f, int E, int k, moe_dtype dtype) {
  if (T < 0 || d < 1 || f < 1 || E < 1 || (k != 1 && k != 2) || k > E) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F16 && dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if ((long long)T * k > 0x7fffffffLL || (long long)T * E > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_F16 && (d % 128 || f % 128)) return MOE_ERR_UNSUPPORTED;
  if (dtype == MOE_F32 && (d % 4 || f % 4)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// ---------------------------------------------------------------- device properties
struct Dev {
  int sms = 0, smem_optin = 0;
};

bool dev_props(Dev* out) {
  static std::mutex mu;
  static Dev cache[64];
  static bool have[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (!have[dev]) {
    Dev p;
    if (cudaDeviceGetAttribute(&p.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&p.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return false;
    cache[dev] = p;
    have[dev] = true;
  }
  *out = cache[dev];
  return true;
}

// ---------------------------------------------------------------- TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D f16 row-major tensor [outer, inner] with a {box_inner, box_outer} box, 128-byte swizzle.
// A descriptor encodes only an address and a geometry, so encoded ones are kept in a small
// per-thread cache keyed by exactly those (a layer called again with the same buffers skips
// the encoding).
struct MapKey {
  const void* ptr;
  uint64_t inner, outer;
  uint32_t bi, bo;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && inner == o.inner && outer == o.outer && bi == o.bi && bo == o.bo;
  }
};
constexpr int kMapCache = 32;
thread_local MapKey t_map_keys[kMapCache];
thread_local CUtensorMap t_maps[kMapCache];
thread_local int t_map_used = 0, t_map_next = 0;

bool encode_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                uint32_t box_inner, uint32_t box_outer);

bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer) {
  const MapKey key{ptr, inner, outer, box_inner, box_outer};
  for (int i = 0; i < t_map_used; ++i)
    if (t_map_keys[i] == key) {
      *m = t_maps[i];
      return true;
    }
  if (!encode_map(m, ptr, inner, outer, box_inner, box_outer)) return false;
  const int slot = t_map_used < kMapCache ? t_map_used++ : (t_map_next++ % kMapCache);
  t_map_keys[slot] = key;
  t_maps[slot] = *m;
  return true;
}

bool encode_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t pow2_at_least(uint32_t v) {
  uint32_t p = 32;
  while (p < v) p <<= 1;
  return p;
}

// Plan of the two tensor-core launches for groups whose tiles hold <= rows_bound rows.
struct TcPlan {
  int nmax, grid, smem_optin;
  uint32_t acc_cols;
};

bool tc_plan(int rows_bound, TcPlan* p) {
  Dev dv;
  if (!dev_props(&dv)) return false;
  p->nmax = std::min(256, std::max(16, (rows_bound + 15) / 16 * 16));
  p->acc_cols = (uint32_t)((p->nmax + 31) / 32 * 32);
  p->grid = dv.sms;
  p->smem_optin = dv.smem_optin;
  return true;
}

// Accumulator slots of the TMEM ring (512 columns, at most 16 slots).
uint32_t slots_for(uint32_t acc_cols) { return std::min(16u, 512u / acc_cols); }

// How an item of mw blocks sits in the slot ring: 2 (room for a whole second item, so the
// epilogue of one item overlaps all of the next item's MMAs), 1 (it fits; with more slots
// than mw the overlap is partial), 0 (does not fit).
int nbuf_for(int mw, uint32_t acc_cols) {
  const uint32_t n = slots_for(acc_cols);
  if (n >= 2u * (uint32_t)mw) return 2;
  if (n >= (uint32_t)mw) return 1;
  return 0;
}

// Weight blocks per item of one GEMM (1, 2 or 4 adjacent 128-row blocks sharing one gather of
// the token rows): the widest that divides every group's M, fits TMEM and three pipeline
// stages, and still leaves about six waves of items.
int choose_mw(long long row_tiles, int M_exp, long long res_tiles, int M_res, const TcPlan& p,
              int E) {
  for (int mw = 4; mw >= 2; mw /= 2) {
    if (M_exp % (128 * mw) || (res_tiles && M_res % (128 * mw))) continue;
    if (nbuf_for(mw, p.acc_cols) == 0) continue;
    if (gemm_stages_for(p.nmax, E, mw, p.smem_optin) < 3) continue;
    const long long items = row_tiles * (M_exp / (128 * mw)) + res_tiles * (M_res / (128 * mw));
    if (items >= 6LL * p.grid) return mw;
  }
  return 1;
}

// Second GEMM: a correction of choose_mw from the row tiles a batch is expected to have
// (the experts that S_rows uniform draws hit, plus tiles for rows beyond one tile each).
// Items of four weight blocks win where they come to 1.5-2 waves (350M+MoE-128 layer:
// T = 512 356.5 -> 338.5 us, T = 4096 407.9 -> 406.2 us per step), not at about one wave
// (T = 128: 258 -> 279 us); where four blocks do not fit TMEM, two beat one from 3.5 waves
// on (PR-MoE E 64 at T = 2048: 993 -> 957 us); and two instead of four where four leave the
// last wave under 90 % full and two fill it at least 10 points better (1.3B+MoE-128 layer,
// Zipf(1.1), T = 8192: 1456 -> 1412 us).  Elsewhere choose_mw's pick stands.
int choose_mw2(int S_rows, int M, long long res_tiles, const TcPlan& p, int E, int picked) {
  auto fits = [&](int mw) {
    return M % (128 * mw) == 0 && nbuf_for(mw, p.acc_cols) > 0 &&
           gemm_stages_for(p.nmax, E, mw, p.smem_optin) >= 3;
  };
  const double hit = E * (1.0 - std::pow(1.0 - 1.0 / E, (double)S_rows));
  const double tiles = std::min<double>(hit, S_rows) +
                       std::max(0.0, S_rows - hit * p.nmax) / p.nmax + (double)res_tiles;
  auto waves = [&](int mw) { return tiles * (M / (128 * mw)) / p.grid; };
  // share of the CTA slots of the last, partly filled wave that have work
  auto fill = [&](int mw) { const double w = waves(mw); return w / std::ceil(w); };
  if (fits(4)) {
    if (waves(4) >= 1.5 && waves(4) <= 2.0) return 4;
    if (picked == 4 && fits(2) && fill(4) < 0.9 && fill(2) >= fill(4) + 0.1) return 2;
  } else if (picked == 1 && fits(2) && waves(2) >= 3.5) {
    return 2;
  }
  return picked;
}

// Decode-sized batches: weight blocks per item (mw) and K chunks per item (ks) together.
// All work units (items x chunks) should run in one round, one per CTA; the widest mw that
// still spreads the weights over at least half the SMs wins (measured: wider items keep more
// bytes in flight per CTA and beat narrower ones that fill every SM), except that a narrower
// mw without K chunks wins over a split one that spreads the weights as widely (the same bytes
// per CTA, and neither fp32 partial sums nor the reduction launch); a chunk keeps at least
// two 64-wide K blocks.  mw candidates must divide every group's M and fit TMEM and three stages.
void choose_split(long long row_tiles, int M_exp, long long res_tiles, int M_res, int nkb_min,
                  const TcPlan& p, int E, int* mw_out, int* ks_out) {
  int best = -1;
  for (int mw = 4; mw >= 1; mw /= 2) {
    if (M_exp % (128 * mw) || (res_tiles && M_res % (128 * mw))) continue;
    if (mw > 1 && (nbuf_for(mw, p.acc_cols) == 0 || gemm_stages_for(p.nmax, E, mw, p.smem_optin) < 3))
      continue;
    const long long items = row_tiles * (M_exp / (128 * mw)) + res_tiles * (M_res / (128 * mw));
    int ks = 1;
    while (ks * 2 <= kMaxSplit && items * ks * 2 <= p.grid && nkb_min / (ks * 2) >= 2) ks *= 2;
    const int score = (int)std::min<long long>(items * ks, p.grid / 2);
    // equal spread: unsplit items win (no fp32 partial sums, no reduction launch); otherwise
    // the widest mw
    if (score > best || (score == best && ks == 1 && *ks_out > 1)) {
      best = score;
      *mw_out = mw;
      *ks_out = ks;
    }
  }
}

// A (M-major weights) descriptor offsets for the 128-byte swizzle layout that two 64-wide
// TMA boxes of 64 K-rows produce: M-blocks 8 KB apart, 8-row K groups 1 KB apart.
constexpr uint32_t kALbo = 8192, kASbo = 1024;

void fill_common(GemmArgs& g, const TcPlan& p, int E, int mw, int* status) {
  memset(&g, 0, sizeof(g));
  g.E = E;
  g.nmax = p.nmax;
  g.mw = mw;
  g.stages = gemm_stages_for(p.nmax, E, mw, p.smem_optin);
  g.acc_cols = p.acc_cols;
  g.nslots = slots_for(p.acc_cols);
  g.tmem_cols = pow2_at_least(g.nslots * p.acc_cols);
  g.a_lbo = kALbo;
  g.a_sbo = kASbo;
  g.status = status;
  g.wait_ns = kDefaultWaitNs;
  g.ksplit = 1;
}

thread_local cudaEvent_t* t_stage_events = nullptr;
thread_local cudaEvent_t t_stage_store[MOE_STAGE_EVENTS];

// Kernels after the first of a call are launched with programmatic dependent launch: each
// starts its prologue while its predecessor drains.  Not while stage events are recorded, so
// that every stage boundary is a full one.
bool use_pdl() { return t_stage_events == nullptr; }

// Inside a stream capture the events are recorded as external event nodes, so that each
// replay of the graph records them (a plain record would only order the capture).
cudaError_t stage_mark(int i, cudaStream_t s) {
  if (!t_stage_events) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t err = cudaStreamIsCapturing(s, &cs);
  if (err != cudaSuccess) return err;
  return cudaEventRecordWithFlags(t_stage_events[i], s,
                                  cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                      : cudaEventRecordDefault);
}

#define MOE_TRY(expr)                          \
  do {                                         \
    cudaError_t e__ = (expr);                  \
    if (e__ != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// Expert FFN stage (both GEMMs) on the tensor cores.
moe_status run_tc_ffn(const void* tokens, const int32_t* perm, const int32_t* offsets,
                      const void* W1, const void* W2, const void* Wr1, const void* Wr2, int T,
                      int d, int f, int E, int f_res, int S_rows, int rows_exp, int rows_bound,
                      __half* H,
                      __half* Hres, int mode, void* out, float* acc32, float* r32,
                      const float* slot_w, const int32_t* drop_slot_of, float* partial,
                      size_t partial_bytes, void* Xg, int* status, bool pdl_first,
                      cudaStream_t s) {
  const bool residual = Wr1 != nullptr;
  const bool pdl = use_pdl();
  // First GEMM.  Where an expert holds at most 64 rows: tiles of at most 64 token rows,
  // gathered through perm by TMA (tile::gather4), so that items can span four weight blocks
  // and each gathered row feeds four MMAs.  Where experts hold more (and the caller gave a
  // buffer Xg of S_rows x d): the kept token rows are first copied to Xg in slot order, and
  // one tile takes all of an expert's rows (up to 256) by 16-row boxes, so that each weight
  // block crosses from L2 to the SM once instead of once per 64-row tile.  Row gathers move
  // 512 bytes per TMA instruction against 2 KB per box, and at these tile heights the gather
  // rate, not HBM, bounded the kernel (2.4B+MoE-128 layer, T = 16384, first GEMM: 4.41 ms with
  // 64-row gathered tiles, 4.95 ms with 160-row gathered tiles).
  const bool pregather = Xg != nullptr && rows_exp > kGather1Rows;
  TcPlan plan1, plan2;
  int rows1 = pregather ? std::min(rows_exp, 256) : std::min(rows_bound, kGather1Rows);
  if (!tc_plan(rows1, &plan1) || !tc_plan(rows_bound, &plan2))
    return MOE_ERR_CUDA;
  const int T_res = residual ? T : 0;
  const int part_rows = S_rows + T_res;
  const long long tiles1 = std::min(E, S_rows) + S_rows / plan1.nmax;
  const long long res1 = residual ? (T + plan1.nmax - 1) / plan1.nmax : 0;
  const long long tiles2 = std::min(E, S_rows) + S_rows / plan2.nmax;
  const long long res2 = residual ? (T + plan2.nmax - 1) / plan2.nmax : 0;
  int mw1 = choose_mw(tiles1, f, res1, f_res, plan1, E);
  int mw2 = choose_mw2(S_rows, d, res2, plan2, E, choose_mw(tiles2, d, res2, d, plan2, E));
  int ks1 = 1, ks2 = 1;
  if (partial) {
    choose_split(tiles1, f, res1, f_res, d / 64, plan1, E, &mw1, &ks1);
    choose_split(tiles2, d, res2, d, residual ? std::min(f, f_res) / 64 : f / 64, plan2, E, &mw2,
                 &ks2);
    const size_t cols1 = std::max(f, residual ? f_res : 0);
    if ((size_t)ks1 * part_rows * cols1 * 4 > partial_bytes) ks1 = 1;
    if ((size_t)ks2 * part_rows * d * 4 > partial_bytes) ks2 = 1;
  }
  CUtensorMap mW1, mX, mWr1, mW2, mH, mWr2, mHres;
  const int S_dim = std::max(S_rows, 1);
  if (!make_map(&mW1, W1, f, (uint64_t)E * d, 64, 64) || !make_map(&mX, tokens, d, T, 64, 1) ||
      !make_map(&mW2, W2, d, (uint64_t)E * f, 64, 64) || !make_map(&mH, H, f, S_dim, 64, 16))
    return MOE_ERR_CUDA;
  if (residual) {
    if (!make_map(&mWr1, Wr1, f_res, d, 64, 64) || !make_map(&mWr2, Wr2, d, f_res, 64, 64) ||
        !make_map(&mHres, Hres, f_res, T, 64, 16))
      return MOE_ERR_CUDA;
  } else {
    mWr1 = mW1;
    mWr2 = mW2;
    mHres = mH;
  }
  GemmArgs g1;
  fill_common(g1, plan1, E, mw1, status);
  if (g1.stages < 2) return MOE_ERR_UNSUPPORTED;
  g1.offsets = offsets;
  g1.perm = perm;
  g1.S_bound = S_rows;
  g1.n_tokens = T;
  g1.n_res_rows = residual ? T : 0;
  g1.K = d;
  g1.K_res = d;
  g1.mt_exp = f / 128 / mw1;
  g1.mt_res = residual ? f_res / 128 / mw1 : 1;
  g1.a_rows_per_expert = d;
  g1.h_out = H;
  g1.ldh = f;
  g1.hres_out = Hres;
  g1.ldhres = f_res;
  if (mode == kModeAccum) {
    g1.zero_buf = acc32;
    g1.zero_bytes = (size_t)T * d * 4;
  } else if (mode == kModeSum) {
    g1.zero_buf = out;                   // the second GEMM adds into it
    g1.zero_bytes = (size_t)T * d * 2;
  }
  if (mode == kModeDirect && drop_slot_of) {
    g1.drop_slot_of = drop_slot_of;
    g1.drop_T = T;
    g1.drop_out = static_cast<__half*>(out);
    g1.drop_d = d;
  }
  g1.ksplit = ks1;
  g1.partial = partial;
  g1.part_rows = part_rows;
  g1.part_cols = std::max(f, residual ? f_res : 0);
  g1.part_res_row0 = S_rows;
  // Larger batches run the residual MLP's first GEMM as a launch of its own: its token rows
  // are contiguous (16-row boxes instead of row gathers) and its tiles take up to 256 rows,
  // where the shared launch would re-stream each dense weight block once per 64-row tile.
  const bool res_apart = residual && ks1 == 1 && T > plan1.nmax;
  if (res_apart) g1.n_res_rows = 0;
  CUtensorMap mXr;                       // tokens by 16-row boxes (contiguous rows)
  if (!make_map(&mXr, tokens, d, T, 64, 16)) return MOE_ERR_CUDA;
  if (pregather) {
    CUtensorMap mXg;
    if (!make_map(&mXg, Xg, d, S_dim, 64, 16)) return MOE_ERR_CUDA;
    MOE_TRY(launch_gather_rows(tokens, perm, offsets, E, S_rows, T, d * 2, Xg, status, s,
                               pdl && pdl_first));
    MOE_TRY(launch_grouped_gemm1_rows(mW1, mXg, mWr1, mXr, g1, plan1.grid, s, pdl));
  } else {
    MOE_TRY(launch_grouped_gemm1(mW1, mX, mWr1, mX, g1, plan1.grid, s, pdl && pdl_first));
  }
  if (ks1 > 1) MOE_TRY(launch_splitk_reduce1(g1, S_rows, T_res, f, f_res, s, pdl));
  if (res_apart) {
    TcPlan planR;
    if (!tc_plan(std::min(T, 256), &planR)) return MOE_ERR_CUDA;
    const long long resR = (T + planR.nmax - 1) / planR.nmax;
    const int mwR = choose_mw(0, f_res, resR, f_res, planR, 0);
    GemmArgs gr;
    fill_common(gr, planR, /*E=*/0, mwR, status);
    if (gr.stages < 2) return MOE_ERR_UNSUPPORTED;
    gr.offsets = offsets;                // no expert group: only offsets[0] (= 0) is read
    gr.perm = perm;
    gr.S_bound = 0;
    gr.n_tokens = T;
    gr.n_res_rows = T;
    gr.K = d;
    gr.K_res = d;
    gr.mt_exp = 1;
    gr.mt_res = f_res / 128 / mwR;
    gr.h_out = H;
    gr.ldh = f;
    gr.hres_out = Hres;
    gr.ldhres = f_res;
    MOE_TRY(launch_grouped_gemm1_rows(mWr1, mXr, mWr1, mXr, gr, planR.grid, s, pdl));
  }
  MOE_TRY(stage_mark(4, s));

  GemmArgs g2;
  fill_common(g2, plan2, E, mw2, status);
  if (g2.stages < 2) return MOE_ERR_UNSUPPORTED;
  g2.offsets = offsets;
  g2.perm = perm;
  g2.S_bound = S_rows;
  g2.n_tokens = T;
  g2.n_res_rows = residual ? T : 0;
  g2.K = f;
  g2.K_res = f_res;
  g2.mt_exp = d / 128 / mw2;
  g2.mt_res = d / 128 / mw2;
  g2.a_rows_per_expert = f;
  g2.mode = mode;
  g2.out = static_cast<__half*>(out);
  g2.acc32 = acc32;
  g2.r32 = r32;
  g2.ldo = d;
  g2.slot_w = slot_w;
  g2.ksplit = ks2;
  g2.partial = partial;
  g2.part_rows = part_rows;
  g2.part_cols = d;
  g2.part_res_row0 = S_rows;
  // Decode-sized batches: the second GEMM's first weight stages load while the first GEMM
  // drains (its offsets come from a kernel at least two launches back: the router or the
  // dispatch, then the first GEMM, or in moe_expert_ffn from the caller).  Measured on the
  // 350M+MoE-128 layer: T = 8 60.7 -> 59.3 us, T = 64 181.5 -> 170.4 us; at larger batches it
  // cost about 1 % (the loads compete with the first GEMM's own stream), so it is off there.
  g2.early_a = pdl && (ks1 > 1 || ks2 > 1);
  MOE_TRY(launch_grouped_gemm2(mW2, mH, mWr2, mHres, g2, plan2.grid, s, pdl));
  if (ks2 > 1) MOE_TRY(launch_splitk_reduce2(g2, S_rows, T_res, d, s, pdl));
  MOE_TRY(stage_mark(5, s));
  return MOE_OK;
}

}  // namespace

namespace moe {

cudaError_t ensure_smem_attr(const void* kernel) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lk(mu);
  if (done.count({kernel, dev})) return cudaSuccess;
  int optin = 0;
  err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  cudaFuncAttributes fa;
  err = cudaFuncGetAttributes(&fa, kernel);
  if (err != cudaSuccess) return err;
  // the limit covers dynamic shared memory only: leave room for the kernel's static part
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes);
  if (err == cudaSuccess) done.insert({kernel, dev});
  return err;
}

// Argument checks of the allocation-free expert FFN (noalloc.cu): those of moe_expert_ffn
// without the workspace.
moe_status expert_ffn_check(const void* tokens, const int32_t* perm, const int32_t* offsets,
                            const void* W1, const void* W2, moe_dtype dtype, int T, int d, int f,
                            int E, int S_max, const void* expert_out) {
  moe_status st = check_shape(T, d, f, E, 1, dtype);
  if (st != MOE_OK) return st;
  if (S_max < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0 || S_max == 0) return MOE_OK;
  if (!tokens || !perm || !offsets || !W1 || !W2 || !expert_out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(tokens) || !aligned16(W1) || !aligned16(W2) || !aligned16(expert_out))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// The expert FFN on a given scratch area holding H [S_max, f]; status may be null.
moe_status expert_ffn_on_scratch(const void* tokens, const int32_t* perm, const int32_t* offsets,
                                 const void* W1, const void* W2, moe_dtype dtype, int T, int d,
                                 int f, int E, int S_max, void* expert_out, uint8_t* scratch,
                                 int* status, cudaStream_t s) {
  if (dtype == MOE_F16) {
    return run_tc_ffn(tokens, perm, offsets, W1, W2, nullptr, nullptr, T, d, f, E, 0, S_max, S_max,
                      S_max, reinterpret_cast<__half*>(scratch), nullptr, kModeExpertOut, expert_out,
                      nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr, status,
                      /*pdl_first=*/false, s);
  }
  SimtArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const float*>(tokens);
  a.offsets = offsets;
  a.perm = perm;
  a.W1 = static_cast<const float*>(W1);
  a.W2 = static_cast<const float*>(W2);
  a.T = T; a.d = d; a.f = f; a.E = E;
  a.S_bound = S_max;
  a.status = status;
  a.H = reinterpret_cast<float*>(scratch);
  a.mode = kModeExpertOut;
  a.out = static_cast<float*>(expert_out);
  MOE_TRY(launch_simt_ffn1(a, S_max, s));
  MOE_TRY(launch_simt_ffn2(a, S_max, s));
  return MOE_OK;
}

}  // namespace moe

extern "C" {

int moe_capacity(int T, int E, float capacity_factor) { return capacity_of(T, E, capacity_factor); }

unsigned long long moe_kernel_launches(void) { return launch_counter().load(); }

moe_status moe_workspace_size(int T, int d, int f, int E, int k, float capacity_factor,
                              moe_mlp_type mlp_type, int f_res, moe_dtype dtype, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_status st = check_shape(T, d, f, E, k, dtype);
  if (st != MOE_OK) return st;
  if (mlp_type != MOE_MLP_STANDARD && mlp_type != MOE_MLP_RESIDUAL) return MOE_ERR_INVALID_ARG;
  const bool residual = mlp_type == MOE_MLP_RESIDUAL;
  if (residual && f_res < 1) return MOE_ERR_INVALID_ARG;
  if (residual && dtype == MOE_F16 && f_res % 128) return MOE_ERR_UNSUPPORTED;
  if (residual && dtype == MOE_F32 && f_res % 4) return MOE_ERR_UNSUPPORTED;
  const int C = capacity_of(T, E, capacity_factor);
  if (C < 0) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(T, d, f, E, k, C, residual, residual ? f_res : 0, dtype == MOE_F16).total;
  return MOE_OK;
}

moe_status moe_gate_topk(const void* tokens, moe_dtype dtype, const float* Wg,
                         const float* logits_in, int T, int d, int E, int k, float* logits_out,
                         float* probs_out, int32_t* topk_idx, float* topk_w, moe_stream_t stream) {
  if (T < 0 || d < 1 || E < 1 || (k != 1 && k != 2) || k > E) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F16 && dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || (long long)T * E > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;                       // empty batch: nothing to read or write
  if (!topk_idx || !topk_w || (!logits_in && (!tokens || !Wg))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(tokens) || !aligned16(Wg) || !aligned16(logits_in) || !aligned16(logits_out) ||
      !aligned16(probs_out) || !aligned16(topk_idx) || !aligned16(topk_w))
    return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (logits_in) {
    MOE_TRY(launch_softmax_topk(logits_in, T, E, k, probs_out, topk_idx, topk_w, logits_out, s));
  } else {
    if (!logits_out) return MOE_ERR_INVALID_ARG;   // the logits need a home
    MOE_TRY(launch_gate_logits(tokens, dtype == MOE_F16, Wg, T, d, E, logits_out, s));
    MOE_TRY(launch_softmax_topk(logits_out, T, E, k, probs_out, topk_idx, topk_w, nullptr, s,
                                use_pdl()));
  }
  return MOE_OK;
}

moe_status moe_dispatch(const int32_t* topk_idx, int T, int E, int k, float capacity_factor,
                        int32_t* counts_raw, int32_t* kept, int32_t* offsets, int32_t* perm,
                        int32_t* slot_of, moe_stream_t stream) {
  if (T < 0 || E < 1 || (k != 1 && k != 2) || k > E) return MOE_ERR_INVALID_ARG;
  const int C = capacity_of(T, E, capacity_factor);
  if (C < 0) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || (long long)T * k > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!topk_idx || !counts_raw || !kept || !offsets || !perm || !slot_of) return MOE_ERR_INVALID_ARG;
  MOE_TRY(launch_dispatch(topk_idx, T, k, E, C, counts_raw, kept, offsets, perm, slot_of, nullptr,
                          nullptr, reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_dispatch_sharded(const int32_t* topk_idx, int T, int E, int k,
                                float capacity_factor, int T_global, const int32_t* counts_all,
                                int n_ranks, int rank, int32_t* counts_raw, int32_t* kept,
                                int32_t* offsets, int32_t* perm, int32_t* slot_of,
                                moe_stream_t stream) {
  if (T < 0 || T_global < T || E < 1 || (k != 1 && k != 2) || k > E) return MOE_ERR_INVALID_ARG;
  if (n_ranks < 1 || rank < 0 || rank >= n_ranks) return MOE_ERR_INVALID_ARG;
  const int C = capacity_of(T_global, E, capacity_factor);
  if (C < 0) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || (long long)T_global * k > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!topk_idx || !counts_raw || !kept || !offsets || !perm || !slot_of) return MOE_ERR_INVALID_ARG;
  if (rank > 0 && !counts_all) return MOE_ERR_INVALID_ARG;
  MOE_TRY(launch_dispatch(topk_idx, T, k, E, C, counts_raw, kept, offsets, perm, slot_of, nullptr,
                          nullptr, reinterpret_cast<cudaStream_t>(stream), false,
                          rank > 0 ? counts_all : nullptr, rank));
  return MOE_OK;
}

moe_status moe_expert_ffn(const void* tokens, const int32_t* perm, const int32_t* offsets,
                          const void* W1, const void* W2, moe_dtype dtype, int T, int d, int f,
                          int E, int S_max, void* expert_out, void* workspace, size_t ws_bytes,
                          moe_stream_t stream) {
  moe_status st = check_shape(T, d, f, E, 1, dtype);
  if (st != MOE_OK) return st;
  if (S_max < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0 || S_max == 0) return MOE_OK;
  if (!tokens || !perm || !offsets || !W1 || !W2 || !expert_out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(tokens) || !aligned16(W1) || !aligned16(W2) || !aligned16(expert_out) ||
      !aligned16(workspace))
    return MOE_ERR_UNSUPPORTED;
  const bool f16 = dtype == MOE_F16;
  if (!workspace || ws_bytes < expert_ffn_ws_bytes(S_max, f, f16)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  MOE_TRY(cudaMemsetAsync(status, 0, sizeof(int), s));
  if (f16) {
    return run_tc_ffn(tokens, perm, offsets, W1, W2, nullptr, nullptr, T, d, f, E, 0, S_max, S_max,
                      S_max, reinterpret_cast<__half*>(ws + kAlign), nullptr, kModeExpertOut, expert_out,
                      nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr, status,
                      /*pdl_first=*/false, s);
  }
  SimtArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const float*>(tokens);
  a.offsets = offsets;
  a.perm = perm;
  a.W1 = static_cast<const float*>(W1);
  a.W2 = static_cast<const float*>(W2);
  a.T = T; a.d = d; a.f = f; a.E = E;
  a.S_bound = S_max;
  a.status = status;
  a.H = reinterpret_cast<float*>(ws + kAlign);
  a.mode = kModeExpertOut;
  a.out = static_cast<float*>(expert_out);
  MOE_TRY(launch_simt_ffn1(a, S_max, s));
  MOE_TRY(launch_simt_ffn2(a, S_max, s));
  return MOE_OK;
}

moe_status moe_combine(const void* expert_out, const int32_t* slot_of, const float* topk_w,
                       const void* residual_in, moe_dtype dtype, int T, int d, int k, void* out,
                       moe_stream_t stream) {
  if (T < 0 || d < 1 || (k != 1 && k != 2)) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F16 && dtype != MOE_F32) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!expert_out || !slot_of || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  MOE_TRY(launch_combine(expert_out, slot_of, topk_w, residual_in, dtype == MOE_F16, T, d, k, out,
                         reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_layer_forward(const void* tokens, const float* Wg, const void* W1, const void* W2,
                             const void* Wr1, const void* Wr2, moe_dtype dtype, int T, int d,
                             int f, int E, int k, float capacity_factor, moe_mlp_type mlp_type,
                             int f_res, void* out, int32_t* topk_idx_out, int32_t* slot_of_out,
                             void* workspace, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_shape(T, d, f, E, k, dtype);
  if (st != MOE_OK) return st;
  if (mlp_type != MOE_MLP_STANDARD && mlp_type != MOE_MLP_RESIDUAL) return MOE_ERR_INVALID_ARG;
  const bool residual = mlp_type == MOE_MLP_RESIDUAL;
  const int C = capacity_of(T, E, capacity_factor);
  if (C < 0) return MOE_ERR_INVALID_ARG;
  if (residual && f_res < 1) return MOE_ERR_INVALID_ARG;
  if (residual && ((dtype == MOE_F16 && f_res % 128) || (dtype == MOE_F32 && f_res % 4)))
    return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;                       // empty batch: nothing to read or write
  if (!tokens || !Wg || !W1 || !W2 || !out) return MOE_ERR_INVALID_ARG;
  if (residual && (!Wr1 || !Wr2)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(tokens) || !aligned16(Wg) || !aligned16(W1) || !aligned16(W2) || !aligned16(out) ||
      !aligned16(workspace) || !aligned16(topk_idx_out) || !aligned16(slot_of_out) ||
      (residual && (!aligned16(Wr1) || !aligned16(Wr2))))
    return MOE_ERR_UNSUPPORTED;
  const bool f16 = dtype == MOE_F16;
  const Ws L = ws_layout(T, d, f, E, k, C, residual, residual ? f_res : 0, f16);
  if (!workspace || ws_bytes < L.total) return MOE_ERR_WORKSPACE;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws + L.status);
  float* logits = reinterpret_cast<float*>(ws + L.logits);
  int32_t* topk_idx = topk_idx_out ? topk_idx_out : reinterpret_cast<int32_t*>(ws + L.topk_idx);
  float* topk_w = reinterpret_cast<float*>(ws + L.topk_w);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* kept = reinterpret_cast<int32_t*>(ws + L.kept);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(ws + L.perm);
  float* slot_w = reinterpret_cast<float*>(ws + L.slot_w);
  int32_t* slot_of = slot_of_out ? slot_of_out : reinterpret_cast<int32_t*>(ws + L.slot_of);
  float* acc32 = L.acc32 ? reinterpret_cast<float*>(ws + L.acc32) : nullptr;
  float* r32 = L.r32 ? reinterpret_cast<float*>(ws + L.r32) : nullptr;
  // top-1 standard: each output row written once; top-2 or one expert plus the residual MLP:
  // two addends summed in place (order-independent); top-2 plus the residual MLP: three
  // addends, summed in fp32 in a fixed order by a finalize pass
  const int mode = (k == 1 && !residual) ? kModeDirect : (k == 2 && residual) ? kModeAccum : kModeSum;
  const int S_max = (int)std::min<long long>((long long)T * k, (long long)E * C);

  // status word and, next to it, the fused router's arrival counter
  unsigned int* route_counter = reinterpret_cast<unsigned int*>(ws + L.status + sizeof(int));
  MOE_TRY(stage_mark(0, s));
  MOE_TRY(cudaMemsetAsync(status, 0, 2 * sizeof(int), s));
  if (f16 && gate_route_small_ok(T, d, E, tokens, Wg)) {
    // decode-sized batch: gate, top-k and dispatch in one launch
    MOE_TRY(launch_gate_route_small(static_cast<const __half*>(tokens), Wg, T, d, E, k, C, logits,
                                    topk_idx, topk_w, counts, kept, offsets, perm, slot_of, slot_w,
                                    route_counter, s));
    MOE_TRY(stage_mark(1, s));
    MOE_TRY(stage_mark(2, s));
  } else {
    MOE_TRY(launch_gate_logits(tokens, f16, Wg, T, d, E, logits, s));
    MOE_TRY(stage_mark(1, s));
    MOE_TRY(launch_softmax_topk(logits, T, E, k, nullptr, topk_idx, topk_w, nullptr, s, use_pdl()));
    MOE_TRY(stage_mark(2, s));
    MOE_TRY(launch_dispatch(topk_idx, T, k, E, C, counts, kept, offsets, perm, slot_of, topk_w,
                            slot_w, s, use_pdl()));
  }
  MOE_TRY(stage_mark(3, s));
  const int rows_exp = std::min(C, T);     // rows of one expert: a token visits it at most once
  const int rows_bound = std::max(rows_exp, residual ? T : 0);
  if (f16) {
    st = run_tc_ffn(tokens, perm, offsets, W1, W2, residual ? Wr1 : nullptr, residual ? Wr2 : nullptr,
                    T, d, f, E, residual ? f_res : 0, S_max, rows_exp, rows_bound,
                    reinterpret_cast<__half*>(ws + L.H),
                    residual ? reinterpret_cast<__half*>(ws + L.Hres) : nullptr, mode, out, acc32, r32,
                    slot_w, k == 1 ? slot_of : nullptr,
                    L.partial_bytes ? reinterpret_cast<float*>(ws + L.partial) : nullptr,
                    L.partial_bytes, L.Xg ? ws + L.Xg : nullptr, status, /*pdl_first=*/true, s);
    if (st != MOE_OK) return st;
  } else {
    SimtArgs a;
    memset(&a, 0, sizeof(a));
    a.x = static_cast<const float*>(tokens);
    a.offsets = offsets;
    a.perm = perm;
    a.W1 = static_cast<const float*>(W1);
    a.W2 = static_cast<const float*>(W2);
    a.Wr1 = residual ? static_cast<const float*>(Wr1) : nullptr;
    a.Wr2 = residual ? static_cast<const float*>(Wr2) : nullptr;
    a.T = T; a.d = d; a.f = f; a.E = E; a.f_res = residual ? f_res : 0;
    a.S_bound = S_max;
    a.status = status;
    a.H = reinterpret_cast<float*>(ws + L.H);
    a.Hres = residual ? reinterpret_cast<float*>(ws + L.Hres) : nullptr;
    a.mode = mode;
    a.out = static_cast<float*>(out);
    a.acc32 = acc32;
    a.r32 = r32;
    a.slot_w = slot_w;
    if (mode == kModeDirect) MOE_TRY(launch_zero_dropped_rows(slot_of, T, k, d, 0, out, s));
    else if (mode == kModeSum) MOE_TRY(launch_zero_f32(static_cast<float*>(out), (size_t)T * d, s));
    else MOE_TRY(launch_zero_f32(acc32, (size_t)T * d, s));
    MOE_TRY(launch_simt_ffn1(a, rows_bound, s));
    MOE_TRY(stage_mark(4, s));
    MOE_TRY(launch_simt_ffn2(a, rows_bound, s));
    MOE_TRY(stage_mark(5, s));
  }
  if (mode == kModeAccum) MOE_TRY(launch_finalize(acc32, r32, T, d, f16, out, s, f16 && use_pdl()));
  MOE_TRY(stage_mark(6, s));
  return MOE_OK;
}

moe_status moe_status_read(const void* workspace, moe_stream_t stream) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = -1;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (v == MOE_OK || v == MOE_ERR_TIMEOUT || v == MOE_ERR_DEVICE_BOUNDS) return (moe_status)v;
  return MOE_ERR_CUDA;
}

const char* moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_set_stage_events(void* const* events, int n_events) {
  if (events == nullptr && n_events == 0) {
    t_stage_events = nullptr;
    return MOE_OK;
  }
  if (events == nullptr || n_events != MOE_STAGE_EVENTS) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < MOE_STAGE_EVENTS; ++i) {
    if (!events[i]) return MOE_ERR_INVALID_ARG;
    t_stage_store[i] = static_cast<cudaEvent_t>(events[i]);
  }
  t_stage_events = t_stage_store;
  return MOE_OK;
}

moe_status moe_selftest_wait(void* workspace, uint64_t timeout_ns, moe_stream_t stream) {
  if (!workspace || timeout_ns < 1 || timeout_ns > 10000000000ull) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  MOE_TRY(cudaMemsetAsync(status, 0, sizeof(int), s));
  MOE_TRY(launch_selftest_wait(status, timeout_ns, s));
  return MOE_OK;
}

}  // extern "C"
