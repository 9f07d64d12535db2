// Internal interface between the C-ABI front end (api.cu) and the kernels.
#pragma once

#include <atomic>
#include <utility>

#include "common.cuh"

namespace moe {

// Kernels this library has enqueued in the process (inside a stream capture: captured).
inline std::atomic<unsigned long long>& launch_counter() {
  static std::atomic<unsigned long long> n{0};
  return n;
}

// Launches `kernel`; with pdl the launch carries programmatic stream serialisation, so the
// grid may start while the previous kernel of the stream finishes (the kernel itself waits
// with pdl_wait() before touching that kernel's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (err == cudaSuccess) launch_counter().fetch_add(1, std::memory_order_relaxed);
  return err;
}

#define MOE_LAUNCH(expr)                     \
  do {                                       \
    const cudaError_t e_ = (expr);           \
    if (e_ != cudaSuccess) return e_;        \
  } while (0)

// Epilogue kinds of the grouped GEMM.
enum : int { kEpiGeluH = 0, kEpiCombine = 1 };
// Output modes of the second GEMM's epilogue (expert tiles).
enum : int {
  kModeDirect = 0,     // out[perm[s]] = f16(w_s * acc): top-1, no residual; each token once
  kModeAccum = 1,      // acc32[perm[s]] += w_s * acc, residual rows to r32, then a finalize
                       // pass (top-2 with the residual MLP: three addends need a fixed order)
  kModeExpertOut = 2,  // out[s] = f16(acc): unscaled rows in slot order (moe_expert_ffn)
  kModeSum = 3         // out[perm[s]] += f16(w_s * acc), residual rows out[t] += f16(acc), into
                       // an output zeroed before: at most two addends per element (top-2, or
                       // one expert plus the residual MLP), so the sum is order-independent
};

struct GemmArgs {
  // groups
  const int32_t* offsets;   // [E + 1] slot offsets per expert, clamped to [0, S_bound] on load
  const int32_t* perm;      // [S] token of each slot
  int E;
  int S_bound;              // rows of H / of the slot-ordered output: no expert row >= it is
                            // read or written, whatever offsets[E] says
  int n_tokens;             // rows of the gathered token matrix (a perm entry must be below)
  int n_res_rows;           // rows of the residual group (T), 0 when absent
  int K, K_res;             // shared dimension of expert / residual tiles
  int mt_exp, mt_res;       // M items (of mw x 128 rows) per expert / residual row tile
  int mw;                   // 128-row weight blocks per item (1, 2 or 4): one TMEM
                            // accumulator each, all fed by the same gathered token rows
  int a_rows_per_expert;    // rows of the A tensor map per expert
  int nmax;                 // rows per tile, multiple of 16, <= 256
  int stages;               // pipeline depth
  uint32_t acc_cols;        // TMEM columns per accumulator (nmax rounded up to 32)
  uint32_t nslots;          // accumulator slots in the TMEM ring (>= mw, <= 16); with more
                            // than mw the epilogue of an item overlaps the next item's MMAs
  uint32_t tmem_cols;       // TMEM columns allocated: power of two >= nslots * acc_cols
  uint32_t a_lbo, a_sbo;    // A (M-major, 128-byte swizzle) descriptor byte offsets
  int mode;                 // kMode* (second GEMM)
  // first GEMM outputs
  __half* h_out;            // [S_max, ldh]
  int ldh;
  __half* hres_out;         // [T, ldhres]
  int ldhres;
  // second GEMM outputs
  __half* out;              // kModeDirect: [T, ldo]; kModeExpertOut: [S_max, ldo]
  float* acc32;             // kModeAccum: [T, ldo]
  float* r32;               // residual tiles: [T, ldo]
  int ldo;
  const float* slot_w;      // [S] gate weight of each slot
  // first GEMM pre-work (epilogue warps, before the first tile)
  void* zero_buf;           // buffer to clear, or null
  size_t zero_bytes;        // its length in bytes (multiple of 16)
  const int32_t* drop_slot_of;  // [T] slot of each token (top-1) for zeroing dropped rows
  int drop_T;
  __half* drop_out;         // out [T, drop_d], or null
  int drop_d;
  // split-K (decode-sized batches): each tile's K range is cut into ksplit chunks run by
  // different CTAs; chunk ks writes fp32 partial sums to partial[ks][prow][part_cols], where
  // prow = row (expert slot) or part_res_row0 + token (residual group); a reduce kernel then
  // sums the chunks in order and applies the epilogue.  ksplit == 1: epilogue in place.
  int ksplit;
  float* partial;
  int part_rows, part_cols, part_res_row0;
  // 1: the offsets come from a kernel at least two launches back (the weights of the first
  // stages are loaded before the wait on the previous kernel)
  int early_a;
  // error reporting
  int* status;
  uint64_t wait_ns;
};

cudaError_t launch_gate_logits(const void* x, int dtype_f16, const float* Wg, int T, int d, int E,
                               float* logits, cudaStream_t s);
cudaError_t launch_softmax_topk(const float* logits, int T, int E, int k, float* probs_out,
                                int32_t* topk_idx, float* topk_w, float* logits_copy,
                                cudaStream_t s, bool pdl = false);
size_t dispatch_smem_bytes(int E);
// Fused gate + top-k + dispatch for T <= 64 (route_small.cu); *counter must be 0 at launch.
bool gate_route_small_ok(int T, int d, int E, const void* x, const void* Wg);
cudaError_t launch_gate_route_small(const __half* x, const float* Wg, int T, int d, int E, int k,
                                    int C, float* logits, int32_t* topk_idx, float* topk_w,
                                    int32_t* counts_raw, int32_t* kept, int32_t* offsets,
                                    int32_t* perm, int32_t* slot_of, float* slot_w,
                                    unsigned int* counter, cudaStream_t s);
cudaError_t launch_dispatch(const int32_t* topk_idx, int T, int k, int E, int C,
                            int32_t* counts_raw, int32_t* kept, int32_t* offsets, int32_t* perm,
                            int32_t* slot_of, const float* topk_w, float* slot_w, cudaStream_t s,
                            bool pdl = false, const int32_t* counts_all = nullptr, int rank = 0);

int gemm_stages_for(int nmax, int E, int mw, int smem_limit);
// Raises the kernel's dynamic shared-memory limit to the device maximum, once per kernel
// and device (host side; launches of any size up to that maximum then need no further call).
cudaError_t ensure_smem_attr(const void* kernel);
cudaError_t launch_grouped_gemm1(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Ar,
                                 const CUtensorMap& Br, const GemmArgs& args, int grid,
                                 cudaStream_t s, bool pdl = false);
cudaError_t launch_grouped_gemm2(const CUtensorMap& A, const CUtensorMap& B, const CUtensorMap& Ar,
                                 const CUtensorMap& Br, const GemmArgs& args, int grid,
                                 cudaStream_t s, bool pdl = false);
// The first GEMM's kernel with contiguous token rows (16-row boxes, no gather): the residual
// MLP's group on its own.
cudaError_t launch_grouped_gemm1_rows(const CUtensorMap& A, const CUtensorMap& B,
                                      const CUtensorMap& Ar, const CUtensorMap& Br,
                                      const GemmArgs& args, int grid, cudaStream_t s,
                                      bool pdl = false);

// fp32 SIMT path (small layers)
struct SimtArgs {
  const float* x;           // [T, d]
  const int32_t* offsets;   // [E + 1]
  const int32_t* perm;      // [S]
  const float* W1;          // [E, d, f]
  const float* W2;          // [E, f, d]
  const float* Wr1;         // [d, f_res] or null
  const float* Wr2;         // [f_res, d]
  int T, d, f, E, f_res;
  int S_bound;              // expert slots are clamped to [0, S_bound) (the S_max of H)
  float* H;                 // [S_max, f]
  float* Hres;              // [T, f_res]
  int mode;                 // kMode*
  float* out;               // kModeDirect: [T, d]; kModeExpertOut: [S_max, d]
  float* acc32;             // kModeAccum: [T, d]
  float* r32;               // residual: [T, d]
  const float* slot_w;
  int* status;              // device status word for MOE_ERR_DEVICE_BOUNDS, or null
};
cudaError_t launch_simt_ffn1(const SimtArgs& a, int S_max, cudaStream_t s);
cudaError_t launch_simt_ffn2(const SimtArgs& a, int S_max, cudaStream_t s);

// elementwise kernels
// Xg[s] = X[perm[s]] for the kept slots s < min(offsets[E], S_bound) (row_bytes % 16 == 0).
cudaError_t launch_gather_rows(const void* X, const int32_t* perm, const int32_t* offsets, int E,
                               int S_bound, int T, int row_bytes, void* Xg, int* status,
                               cudaStream_t s, bool pdl = false);
cudaError_t launch_zero_f32(float* p, size_t n, cudaStream_t s);
cudaError_t launch_zero_dropped_rows(const int32_t* slot_of, int T, int k, int d, int dtype_f16,
                                     void* out, cudaStream_t s);
cudaError_t launch_finalize(const float* acc32, const float* r32, int T, int d, int dtype_f16,
                            void* out, cudaStream_t s, bool pdl = false);
cudaError_t launch_combine(const void* expert_out, const int32_t* slot_of, const float* topk_w,
                           const void* residual_in, int dtype_f16, int T, int d, int k, void* out,
                           cudaStream_t s);
cudaError_t launch_selftest_wait(int* status, uint64_t timeout_ns, cudaStream_t s);
// split-K reductions (fixed chunk order): first GEMM -> GeLU -> H / Hres; second GEMM -> the
// combine of the given mode / r32
cudaError_t launch_splitk_reduce1(const GemmArgs& g, int S_max, int T_res, int f, int f_res,
                                  cudaStream_t s, bool pdl = false);
cudaError_t launch_splitk_reduce2(const GemmArgs& g, int S_max, int T_res, int d, cudaStream_t s,
                                  bool pdl = false);

}  // namespace moe
