// attn_kernel.h -- parameters shared by the host launcher and the sm_103a
// attention kernels (one instantiation per head dimension and mask kind).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

constexpr int kBM = 128;        // query rows per Q tile: one TMEM lane and one softmax thread per row
constexpr int kBN = 128;        // keys per K/V tile
constexpr int kWarps = 12;      // warpgroup 0: warp 0 loader, warp 1 MMA issuer (warps 2-3 idle);
                                // warpgroups 1 / 2: softmax of Q tile 0 / 1
constexpr int kRegsControl = 72;   // registers per thread of warpgroup 0 after setmaxnreg
constexpr int kRegsSoftmax = 216;  // registers per thread of warpgroups 1-2 after setmaxnreg
// 128 * kRegsControl + 256 * kRegsSoftmax must not exceed 384 * 168 (the launch's registers)
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= 384 * 168, "register split");
constexpr int kThreads = kWarps * 32;
constexpr float kRescaleLog2 = 8.0f;  // keep a stale row maximum until the true one exceeds it by 2^8
constexpr int kMaxSplitCtas = 256;  // largest grid of the split schedule (its range table lives in shared memory)

// Mask specialisations (the C-ABI's NA2D splits into clamp and wrap here).
// Kernel variants. Neighbourhood masks are kMaskNa plus flags: which axes
// wrap (rows, columns) and whether the windows are dilated, so that each
// combination compiles to its own arithmetic (dilation 1 keeps intervals).
// Volumes (3-D windows) are one further variant, kMaskNa3, that reads the
// wrap choice of each axis and the dilation at run time.
enum MaskKind : int { kMaskNone = 0, kMaskCausal = 1, kMaskNa = 2 };
constexpr int kNaWrapCols = 1, kNaWrapRows = 2, kNaDilated = 4;
constexpr int kMaskNa3 = kMaskNa + 8;
// Bottom-right causal: causal with the key bound shifted by Nk - Nq (read at
// run time), kept apart so that top-left causal keeps a compile-time bound.
constexpr int kMaskCausalBR = kMaskNa3 + 1;
constexpr int kMaskKinds = kMaskCausalBR + 1;
constexpr int kNa3WrapCols = 1, kNa3WrapRows = 2, kNa3WrapDepth = 4;  // KernelParams::na_wrap
__host__ __device__ constexpr int na_mask(bool wrap_rows, bool wrap_cols, bool dilated) {
  return kMaskNa + (wrap_cols ? kNaWrapCols : 0) + (wrap_rows ? kNaWrapRows : 0) +
         (dilated ? kNaDilated : 0);
}
__host__ __device__ constexpr bool mask_is_na(int m) { return m >= kMaskNa && m <= kMaskNa3; }
__host__ __device__ constexpr bool mask_is_causal(int m) { return m == kMaskCausal || m == kMaskCausalBR; }
__host__ __device__ constexpr bool mask_is_na2(int m) { return m >= kMaskNa && m < kMaskNa3; }
__host__ __device__ constexpr bool mask_na_wrap_rows(int m) {
  return mask_is_na2(m) && ((m - kMaskNa) & kNaWrapRows) != 0;
}
__host__ __device__ constexpr bool mask_na_wrap_cols(int m) {
  return mask_is_na2(m) && ((m - kMaskNa) & kNaWrapCols) != 0;
}
__host__ __device__ constexpr bool mask_na_dilated(int m) {
  return mask_is_na2(m) && ((m - kMaskNa) & kNaDilated) != 0;
}

// Roles recorded in the device status word when a bounded wait runs out.
enum Role : uint32_t { kRoleLoader = 0, kRoleMma = 1, kRoleSoftmax = 2 };

struct KernelParams {
  CUtensorMap tm_q;             // 4-D (d, n, h, b) bf16 maps, box (swizzle span, 128, 1, 1)
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  void* o;                      // bf16 output
  float* lse;                   // fp32 [B, H, Nq] or nullptr
  int64_t o_sb, o_sh, o_sn;     // element strides of O for b, h, n
  int B, H, Nq, Nk;
  float c;                      // scale * log2(e): scores enter exp2 in log2 units
  int grid_h, grid_w;           // neighbourhood masks only: token grid
  int window_h, window_w;       // window size along the rows and the columns
  int dilation;                 // neighbourhood masks: key stride along each axis (>= 1)
  int causal_off;               // kMaskCausalBR: key k allowed iff k <= q + causal_off (Nk - Nq)
  int grid_d, window_d;         // kMaskNa3: depth of the volume and window along it
  int na_wrap;                  // kMaskNa3: kNa3Wrap* bits of the axes that wrap
  int q_tiles;                  // Q tiles (of 128 rows) per task: 2, or 1 when a launch has
                                // fewer pairs than persistent CTAs
  int twin;                     // neighbourhood masks with q_tiles == 1: both softmax warpgroups
                                // on the one Q tile, its K/V tiles taken in turn (set at launch)
  int n_qtasks;                 // ceil(Nq / (128 * q_tiles)): tasks per (batch, head)
  int n_kv;                     // ceil(Nk / 128)
  int n_tasks;                  // B * H * n_qtasks
  // Work split. split == 0: whole tasks, round robin over the CTAs. split == 1
  // (unmasked only): the tasks' K/V tiles form one sequence of `units`
  // (task-major) and CTA c takes units [c*units/G, (c+1)*units/G); a task cut
  // between CTAs leaves partial results in the workspace and the last part to
  // finish merges them.
  int split;
  int64_t units;
  float* ws_part;               // per CTA 2 slots x 2 Q tiles x 128 rows x (d + 2) fp32
  unsigned long long* ws_count; // per (task, Q tile, 32-row quarter): epoch << 32 | parts arrived
  uint32_t epoch;               // this call's tag in ws_count (never 0)
  uint64_t timeout_ns;          // bound on every mbarrier wait
  int inject;                   // 1: loader withholds one K tile (tests the bounded wait)
  uint32_t* status;             // device status word: code, role, tile, CTA
};

// Backward pass: the forward's parameters (maps of Q, K, V, shapes, masks,
// status) plus dO and the gradients (all bf16 contiguous [B, H, N, d]).
struct BwdParams {
  KernelParams f;               // f.c = scale * log2(e)
  CUtensorMap tm_do;            // dO, the same map shape as Q
  const void* o;                // forward output
  const void* dout;
  const float* lse;             // forward log-sum-exp, natural log, [B, H, Nq]
  float* dd;                    // scratch [B, H, Nq]: rowsum(dO * O)
  void* dq;
  void* dk;
  void* dv;
  float scale;
};

// Per-head-dimension launchers, defined in attn_fwd_d{32,64,128}.cu.
cudaError_t launch_d32(const KernelParams& p, int mask, int grid, cudaStream_t s);
cudaError_t launch_d64(const KernelParams& p, int mask, int grid, cudaStream_t s);
// Backward launchers (D = rowsum(dO * O), dQ, then dK and dV), in attn_bwd.cu.
// The dQ and the dK/dV kernels are independent: dK/dV runs on `aux`, forked
// from s after D and joined back into s.
cudaError_t launch_bwd(const BwdParams& p, int d, int mask, cudaStream_t s, cudaStream_t aux,
                       cudaEvent_t fork, cudaEvent_t join);
cudaError_t launch_d128(const KernelParams& p, int mask, int grid, cudaStream_t s);
// 1 if a launch of kernel variant `mask` with these parameters should run its
// tasks as twins (KernelParams::twin), else 0; in attn_fwd_d64.cu.
int twin_tasks(const KernelParams& p, int mask);

}  // namespace attn
