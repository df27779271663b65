// attn_host.cu -- the C ABI of libattn.so (declared in include/attn.h).
//
// Host work per call: validate the arguments (before any CUDA call), encode
// the three TMA tensor maps, pick the kernel specialisation, launch once on
// the caller's stream. The device memory the library owns: one status word
// per device, and a workspace for split schedules, both allocated on first
// use (the workspace grows when a call needs more).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "attn_kernel.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

thread_local cudaStream_t t_stream = nullptr;
thread_local char t_err[512] = {0};

struct DeviceState {
  uint32_t* status = nullptr;  // 4 x u32 device status word
  int sm_count = 0;
  void* ws = nullptr;          // workspace of split schedules (zero-filled when allocated)
  size_t ws_bytes = 0;
  uint32_t epoch = 0;          // tag of the last split call
  float* dd = nullptr;         // backward scratch: rowsum(dO * O), grown when too small
  size_t dd_bytes = 0;
  cudaStream_t aux = nullptr;  // backward: second stream (dK/dV beside dQ) and its events
  cudaEvent_t fork = nullptr, join = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t align256(size_t x) { return (x + 255) & ~size_t{255}; }

constexpr int64_t kMinSplitUnits = 4;

// How a call's work is laid out over the persistent CTAs.
struct Plan {
  int grid = 0;
  int split = 0;
  int q_tiles = 2, n_qtasks = 0, n_kv = 0, n_tasks = 0;
  int64_t units = 0;
  size_t part_bytes = 0, count_bytes = 0;
  size_t ws_bytes() const { return split ? align256(part_bytes) + align256(count_bytes) : 0; }
};

int make_plan(const attn_params_ex* p, int sm_count, Plan* pl) {
  int ctas = sm_count;
  if (p->num_ctas > 0 && p->num_ctas < ctas) ctas = p->num_ctas;
  // A task is a pair of Q tiles, whose softmax warpgroups take turns on the
  // tensor core; a masked launch with fewer pairs than CTAs (small or
  // neighbourhood problems, never split) gives each task one Q tile instead,
  // so that twice as many SMs work, each on a shorter chain.
  const int pairs = p->B * p->H * ((p->Nq + 2 * attn::kBM - 1) / (2 * attn::kBM));
  pl->q_tiles = (p->mask_kind != ATTN_MASK_NONE && pairs < ctas) ? 1 : 2;
  pl->n_qtasks = (p->Nq + pl->q_tiles * attn::kBM - 1) / (pl->q_tiles * attn::kBM);
  pl->n_kv = (p->Nk + attn::kBN - 1) / attn::kBN;
  pl->n_tasks = p->B * p->H * pl->n_qtasks;
  pl->units = static_cast<int64_t>(pl->n_tasks) * pl->n_kv;
  if (p->schedule == 2 && p->mask_kind != ATTN_MASK_NONE)
    return fail(ATTN_ERR_INVALID_ARG, "schedule 2 applies to ATTN_MASK_NONE only");
  pl->split = p->schedule == 2 ||
              (p->schedule == 0 && p->mask_kind == ATTN_MASK_NONE && pl->n_tasks % ctas != 0);
  if (pl->split) {
    // at least kMinSplitUnits K/V tiles per CTA: fewer, larger parts to merge
    const int64_t by_units = (pl->units + kMinSplitUnits - 1) / kMinSplitUnits;
    pl->grid = static_cast<int>(by_units < ctas ? by_units : ctas);
    if (pl->grid > attn::kMaxSplitCtas) pl->grid = attn::kMaxSplitCtas;
    // the kernel counts a CTA's share in 32 bits: larger shares run as whole tasks
    if ((pl->units + pl->grid - 1) / pl->grid >= (int64_t{1} << 31)) pl->split = 0;
  }
  if (pl->split) {
    pl->part_bytes = static_cast<size_t>(pl->grid) * 2 * 2 * 128 * (p->d + 2) * sizeof(float);
    pl->count_bytes = static_cast<size_t>(pl->n_tasks) * 2 * 4 * sizeof(unsigned long long);
  } else {
    pl->grid = pl->n_tasks < ctas ? pl->n_tasks : ctas;
  }
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t isqrt64(int64_t n) {
  int64_t r = static_cast<int64_t>(std::sqrt(static_cast<double>(n)));
  while (r * r > n) --r;
  while ((r + 1) * (r + 1) <= n) ++r;
  return r;
}

// Host-only argument checks; fills the derived grid and strides.
struct Checked {
  int grid_h = 0, grid_w = 0, grid_d = 0;
  int64_t qs[3], ks[3], vs[3], os[3];
};

int check_strides(const int64_t in[3], int64_t out[3], int64_t N, int64_t H, int64_t d,
                  const char* name) {
  if (in[0] == 0 && in[1] == 0 && in[2] == 0) {
    out[2] = d;
    out[1] = N * d;
    out[0] = H * N * d;
    return ATTN_OK;
  }
  for (int i = 0; i < 3; ++i) {
    if (in[i] <= 0) return fail(ATTN_ERR_INVALID_ARG, "%s stride %d must be positive", name, i);
    if (in[i] % 8 != 0)
      return fail(ATTN_ERR_MISALIGNED, "%s stride %d (%lld elements) is not a multiple of 8", name,
                  i, static_cast<long long>(in[i]));
    out[i] = in[i];
  }
  if (out[2] < d) return fail(ATTN_ERR_INVALID_ARG, "%s row stride is smaller than d", name);
  return ATTN_OK;
}

int validate(const attn_params_ex* p, Checked* c) {
  if (p == nullptr) return fail(ATTN_ERR_INVALID_ARG, "null parameter block");
  if (p->B < 1 || p->H < 1 || p->Nq < 1 || p->Nk < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, Nq, Nk must be >= 1 (got %d, %d, %d, %d)", p->B,
                p->H, p->Nq, p->Nk);
  if (p->d < 1) return fail(ATTN_ERR_INVALID_ARG, "d must be >= 1");
  if (p->d != 32 && p->d != 64 && p->d != 128)
    return fail(ATTN_ERR_UNSUPPORTED, "head dimension %d is not one of 32, 64, 128", p->d);
  if (!std::isfinite(p->scale) || !(p->scale > 0.f))
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (p->mask_kind < ATTN_MASK_NONE || p->mask_kind > ATTN_MASK_CAUSAL_BR)
    return fail(ATTN_ERR_INVALID_ARG, "unknown mask kind %d", p->mask_kind);
  const int64_t BH = static_cast<int64_t>(p->B) * p->H;
  const int64_t n_qtiles = (static_cast<int64_t>(p->Nq) + attn::kBM - 1) / attn::kBM;
  if (BH * n_qtiles >= (int64_t{1} << 31))
    return fail(ATTN_ERR_INVALID_ARG, "too many (batch, head, query-tile) tasks");
  const bool na3 = p->mask_kind == ATTN_MASK_NA3D;
  if (!na3 && (p->grid_d != 0 || p->window_d != 0 || p->wrap_d != 0))
    return fail(ATTN_ERR_INVALID_ARG, "grid_d/window_d/wrap_d apply to NA3D only (need 0)");
  if (p->mask_kind != ATTN_MASK_NA2D && !na3) {
    if (p->window != 0 || p->window_w != 0 || p->dilation != 1 || p->wrap != 0 ||
        p->grid_h != 0 || p->grid_w != 0)
      return fail(ATTN_ERR_INVALID_ARG,
                  "window/dilation/wrap/grid apply to NA2D and NA3D only (need 0/1/0/0x0)");
  } else {
    if (p->wrap < 0 || p->wrap > 3)
      return fail(ATTN_ERR_INVALID_ARG, "wrap must be 0 (none), 1 (both axes), 2 (rows) or 3 "
                  "(columns)");
    if (p->window < 1 || p->window % 2 == 0)
      return fail(ATTN_ERR_INVALID_ARG, "window must be odd and >= 1 (got %d)", p->window);
    if (p->window_w != 0 && (p->window_w < 1 || p->window_w % 2 == 0))
      return fail(ATTN_ERR_INVALID_ARG, "window_w must be 0 or odd and >= 1 (got %d)",
                  p->window_w);
    if (p->dilation < 1) return fail(ATTN_ERR_INVALID_ARG, "dilation must be >= 1");
    if (p->Nq != p->Nk) return fail(ATTN_ERR_INVALID_ARG, "neighbourhood masks need Nq == Nk");
    if (na3) {
      if (p->wrap_d != 0 && p->wrap_d != 1) return fail(ATTN_ERR_INVALID_ARG, "wrap_d must be 0 or 1");
      if (p->window_d != 0 && (p->window_d < 1 || p->window_d % 2 == 0))
        return fail(ATTN_ERR_INVALID_ARG, "window_d must be 0 or odd and >= 1 (got %d)",
                    p->window_d);
      if (p->grid_d < 1 || p->grid_h < 1 || p->grid_w < 1 ||
          static_cast<int64_t>(p->grid_d) * p->grid_h * p->grid_w != p->Nq)
        return fail(ATTN_ERR_INVALID_ARG, "NA3D volume %dx%dx%d does not hold Nq=%d tokens",
                    p->grid_d, p->grid_h, p->grid_w, p->Nq);
      const int kd = p->window_d ? p->window_d : p->window;
      if (kd > 1 && static_cast<int64_t>(kd) * p->dilation > p->grid_d)
        return fail(ATTN_ERR_INVALID_ARG, "window_d*dilation (%lld) exceeds the depth %d",
                    static_cast<long long>(kd) * p->dilation, p->grid_d);
      c->grid_d = p->grid_d;
      c->grid_h = p->grid_h;
      c->grid_w = p->grid_w;
    } else if (p->grid_h == 0 && p->grid_w == 0) {
      const int64_t g = isqrt64(p->Nq);
      if (g * g != p->Nq)
        return fail(ATTN_ERR_INVALID_ARG, "NA2D with Nq=%d needs a square grid or grid_h/grid_w",
                    p->Nq);
      c->grid_h = c->grid_w = static_cast<int>(g);
    } else {
      if (p->grid_h < 1 || p->grid_w < 1 ||
          static_cast<int64_t>(p->grid_h) * p->grid_w != p->Nq)
        return fail(ATTN_ERR_INVALID_ARG, "grid %dx%d does not hold Nq=%d tokens", p->grid_h,
                    p->grid_w, p->Nq);
      c->grid_h = p->grid_h;
      c->grid_w = p->grid_w;
    }
    const int64_t span_h = static_cast<int64_t>(p->window) * p->dilation;
    const int64_t span_w = static_cast<int64_t>(p->window_w ? p->window_w : p->window) * p->dilation;
    // a window of 1 holds only the query, whatever the dilation
    if ((p->window > 1 && span_h > c->grid_h) ||
        ((p->window_w ? p->window_w : p->window) > 1 && span_w > c->grid_w))
      return fail(ATTN_ERR_INVALID_ARG,
                  "window*dilation (%lld rows, %lld columns) exceeds the %dx%d grid",
                  static_cast<long long>(span_h), static_cast<long long>(span_w), c->grid_h,
                  c->grid_w);
  }
  if (!p->q || !p->k || !p->v || !p->o)
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-null");
  if (!aligned16(p->q) || !aligned16(p->k) || !aligned16(p->v) || !aligned16(p->o))
    return fail(ATTN_ERR_MISALIGNED, "q, k, v and o must be 16-byte aligned");
  if (p->lse && (reinterpret_cast<uintptr_t>(p->lse) & 3u))
    return fail(ATTN_ERR_MISALIGNED, "lse must be 4-byte aligned");
  if (p->num_ctas < 0) return fail(ATTN_ERR_INVALID_ARG, "num_ctas must be >= 0");
  if (p->inject != 0 && p->inject != 1) return fail(ATTN_ERR_INVALID_ARG, "inject must be 0 or 1");
  if (p->schedule < 0 || p->schedule > 2)
    return fail(ATTN_ERR_INVALID_ARG, "schedule must be 0, 1 or 2");
  if (p->workspace && !aligned16(p->workspace))
    return fail(ATTN_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  if (static_cast<int64_t>(p->B) * p->H * ((p->Nq + 255) / 256) * ((p->Nk + 127) / 128) >=
      (int64_t{1} << 40))
    return fail(ATTN_ERR_INVALID_ARG, "problem too large");
  int rc;
  if ((rc = check_strides(p->q_stride, c->qs, p->Nq, p->H, p->d, "q")) != ATTN_OK) return rc;
  if ((rc = check_strides(p->k_stride, c->ks, p->Nk, p->H, p->d, "k")) != ATTN_OK) return rc;
  if ((rc = check_strides(p->v_stride, c->vs, p->Nk, p->H, p->d, "v")) != ATTN_OK) return rc;
  if ((rc = check_strides(p->o_stride, c->os, p->Nq, p->H, p->d, "o")) != ATTN_OK) return rc;
  return ATTN_OK;
}

// Kernel mask variant of a validated problem; fills the neighbourhood fields of kp.
int kernel_mask(const attn_params_ex* p, const Checked& c, attn::KernelParams* kp) {
  const bool na = p->mask_kind == ATTN_MASK_NA2D || p->mask_kind == ATTN_MASK_NA3D;
  const bool wrap_rows = p->wrap == 1 || p->wrap == 2, wrap_cols = p->wrap == 1 || p->wrap == 3;
  kp->grid_h = c.grid_h;
  kp->grid_w = c.grid_w;
  kp->grid_d = c.grid_d;
  kp->window_h = p->window;
  kp->window_w = p->window_w ? p->window_w : p->window;
  kp->window_d = p->window_d ? p->window_d : p->window;
  kp->dilation = na ? p->dilation : 1;
  kp->na_wrap = (wrap_cols ? attn::kNa3WrapCols : 0) | (wrap_rows ? attn::kNa3WrapRows : 0) |
                (p->wrap_d ? attn::kNa3WrapDepth : 0);
  kp->causal_off = p->mask_kind == ATTN_MASK_CAUSAL_BR ? p->Nk - p->Nq : 0;
  switch (p->mask_kind) {
    case ATTN_MASK_CAUSAL: return attn::kMaskCausal;
    case ATTN_MASK_CAUSAL_BR: return attn::kMaskCausalBR;
    case ATTN_MASK_NA2D: return attn::na_mask(wrap_rows, wrap_cols, p->dilation > 1);
    case ATTN_MASK_NA3D: return attn::kMaskNa3;
    default: return attn::kMaskNone;
  }
}

int get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return ATTN_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDriverEntryPointByVersion");
  if (q != cudaDriverEntryPointSuccess || fn == nullptr)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return ATTN_OK;
}

// Per-device state; creates the status word on first use.
int device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device ordinal %d out of range", dev);
  // make the device's primary context current on this thread: the tensor-map
  // encoder is a driver call, and a thread may not have touched CUDA yet
  // (e.g. an autograd worker thread)
  if ((e = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& s = g_dev[dev];
  if (s.status == nullptr) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
      return fail(ATTN_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                  dev, major, minor);
    if ((e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    void* ptr = nullptr;
    if ((e = cudaMalloc(&ptr, 4 * sizeof(uint32_t))) != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    if ((e = cudaMemset(ptr, 0, 4 * sizeof(uint32_t))) != cudaSuccess) {
      cudaFree(ptr);
      return cuda_fail(e, "cudaMemset");
    }
    s.status = static_cast<uint32_t*>(ptr);
  }
  *out = &s;
  return ATTN_OK;
}

// 4-D bf16 tensor map over (d, n, h, b), box (box_cols, 128, 1, 1).
int encode_map(CUtensorMap* m, const void* base, int d, int N, int H, int B, const int64_t st[3],
               int box_cols, CUtensorMapSwizzle swz, const char* name) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st[2]) * 2, static_cast<cuuint64_t>(st[1]) * 2,
                           static_cast<cuuint64_t>(st[0]) * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(attn::kBN), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name,
                static_cast<int>(r));
  return ATTN_OK;
}

// The kernel parameters of a validated call: tensor maps, output and shapes,
// the mask fields (returns the kernel's mask variant in *mask), the plan's
// schedule and the timeout and test hook. Workspace, epoch and status are
// left for the caller (the regular and the no-alloc entry points differ
// there and only there).
int fill_params(const attn_params_ex* p, const Checked& c, const Plan& pl, attn::KernelParams* kp,
                int* mask) {
  std::memset(kp, 0, sizeof(*kp));
  const int box_cols = p->d >= 64 ? 64 : 32;
  const CUtensorMapSwizzle swz = p->d >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  int rc;
  if ((rc = encode_map(&kp->tm_q, p->q, p->d, p->Nq, p->H, p->B, c.qs, box_cols, swz, "q")) != ATTN_OK ||
      (rc = encode_map(&kp->tm_k, p->k, p->d, p->Nk, p->H, p->B, c.ks, box_cols, swz, "k")) != ATTN_OK ||
      (rc = encode_map(&kp->tm_v, p->v, p->d, p->Nk, p->H, p->B, c.vs, box_cols, swz, "v")) != ATTN_OK)
    return rc;
  kp->o = p->o;
  kp->lse = p->lse;
  kp->o_sb = c.os[0];
  kp->o_sh = c.os[1];
  kp->o_sn = c.os[2];
  kp->B = p->B;
  kp->H = p->H;
  kp->Nq = p->Nq;
  kp->Nk = p->Nk;
  kp->c = p->scale * 1.4426950408889634f;
  *mask = kernel_mask(p, c, kp);
  kp->q_tiles = pl.q_tiles;
  kp->n_qtasks = pl.n_qtasks;
  kp->n_kv = pl.n_kv;
  kp->n_tasks = pl.n_tasks;
  kp->split = pl.split;
  kp->units = pl.units;
  kp->timeout_ns = p->timeout_ns ? p->timeout_ns : kDefaultTimeoutNs;
  kp->inject = p->inject;
  kp->twin = attn::twin_tasks(*kp, *mask);
  return ATTN_OK;
}

// ATTN_LOG=1 in the environment: one line on stderr per launch, naming the
// kernel specialisation and the schedule.
bool log_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("ATTN_LOG");
    return e != nullptr && e[0] != '\0' && e[0] != '0';
  }();
  return on;
}

const char* mask_name(int mask_kind) {
  switch (mask_kind) {
    case ATTN_MASK_NONE: return "none";
    case ATTN_MASK_CAUSAL: return "causal";
    case ATTN_MASK_CAUSAL_BR: return "causal_br";
    case ATTN_MASK_NA2D: return "na2d";
    case ATTN_MASK_NA3D: return "na3d";
    default: return "?";
  }
}

void log_launch(const char* entry, const attn_params_ex* p, const attn::KernelParams& kp, int mask,
                const Plan& pl) {
  if (!log_enabled()) return;
  std::fprintf(stderr,
               "%s: d=%d mask=%s variant=%d B=%d H=%d Nq=%d Nk=%d grid_hw=%dx%d window=%dx%d "
               "dilation=%d wrap=%d schedule=%s grid=%d tasks=%d units=%lld q_tiles=%d twin=%d\n",
               entry, p->d, mask_name(p->mask_kind), mask, p->B, p->H, p->Nq, p->Nk, kp.grid_h,
               kp.grid_w, kp.window_h, kp.window_w, kp.dilation, kp.na_wrap,
               pl.split ? "split" : "whole", pl.grid, pl.n_tasks, static_cast<long long>(pl.units),
               kp.q_tiles, kp.twin);
}

// Device pointers of the call's workspace: the caller's, or the library's own
// (grown, and zero-filled, when too small). Also hands out the call's epoch.
int acquire_workspace(const attn_params_ex* p, const Plan& pl, DeviceState* ds, void** ws,
                      uint32_t* epoch) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (++ds->epoch == 0) ds->epoch = 1;
  *epoch = ds->epoch;
  const size_t need = pl.ws_bytes();
  if (p->workspace) {
    if (p->workspace_bytes < need)
      return fail(ATTN_ERR_INVALID_ARG, "workspace of %llu bytes, this call needs %zu",
                  static_cast<unsigned long long>(p->workspace_bytes), need);
    *ws = p->workspace;
    return ATTN_OK;
  }
  if (ds->ws_bytes < need) {
    cudaError_t e;
    if (ds->ws) {
      if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
      cudaFree(ds->ws);
      ds->ws = nullptr;
      ds->ws_bytes = 0;
    }
    void* ptr = nullptr;
    if ((e = cudaMalloc(&ptr, need)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
    if ((e = cudaMemset(ptr, 0, need)) != cudaSuccess) {
      cudaFree(ptr);
      return cuda_fail(e, "cudaMemset(workspace)");
    }
    ds->ws = ptr;
    ds->ws_bytes = need;
  }
  *ws = ds->ws;
  return ATTN_OK;
}

// Reads and clears the no-alloc entry point's status word on device `dev`
// (zeros if that entry point was not used there), and forgets its per-device
// state (under g_mu); defined with it below.
int noalloc_take_status(int dev, uint32_t word[4]);
void noalloc_forget();

}  // namespace

extern "C" {

void attn_params_init(attn_params_ex* p) {
  if (!p) return;
  std::memset(p, 0, sizeof(*p));
  p->dilation = 1;
}

int attn_fwd_ex(const attn_params_ex* p) {
  t_err[0] = 0;
  Checked c;
  int rc = validate(p, &c);
  if (rc != ATTN_OK) return rc;
  if ((rc = get_encoder()) != ATTN_OK) return rc;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != ATTN_OK) return rc;
  Plan pl;
  if ((rc = make_plan(p, ds->sm_count, &pl)) != ATTN_OK) return rc;
  attn::KernelParams kp;
  int mask = 0;
  if ((rc = fill_params(p, c, pl, &kp, &mask)) != ATTN_OK) return rc;
  if (pl.split) {
    void* ws = nullptr;
    if ((rc = acquire_workspace(p, pl, ds, &ws, &kp.epoch)) != ATTN_OK) return rc;
    kp.ws_part = static_cast<float*>(ws);
    kp.ws_count = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) +
                                                         align256(pl.part_bytes));
  }
  kp.status = ds->status;
  log_launch("attn_fwd", p, kp, mask, pl);

  cudaStream_t s = p->stream ? static_cast<cudaStream_t>(p->stream) : t_stream;
  cudaError_t e;
  if (p->ev_start && (e = cudaEventRecord(static_cast<cudaEvent_t>(p->ev_start), s)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord(start)");
  switch (p->d) {
    case 32: e = attn::launch_d32(kp, mask, pl.grid, s); break;
    case 64: e = attn::launch_d64(kp, mask, pl.grid, s); break;
    default: e = attn::launch_d128(kp, mask, pl.grid, s); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  if (p->ev_stop && (e = cudaEventRecord(static_cast<cudaEvent_t>(p->ev_stop), s)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord(stop)");
  return ATTN_OK;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
             int Nk, int d, float scale, int mask_kind, int window, int dilation, int wrap) {
  attn_params_ex p;
  attn_params_init(&p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.d = d;
  p.scale = scale;
  p.mask_kind = mask_kind;
  p.window = window;
  p.dilation = dilation;
  p.wrap = wrap;
  return attn_fwd_ex(&p);
}

int attn_set_stream(void* stream) {
  t_stream = static_cast<cudaStream_t>(stream);
  return ATTN_OK;
}

int attn_get_device_status(uint32_t* detail) {
  t_err[0] = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device ordinal %d out of range", dev);
  // Reads the status words that exist on this device and allocates nothing:
  // the library's own (created by the first attn_fwd_ex or attn_bwd) and the
  // no-alloc entry point's (inside its fixed array). The first failure wins.
  uint32_t* status = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    status = g_dev[dev].status;
  }
  uint32_t word[4] = {0, 0, 0, 0};
  if (status != nullptr) {
    if ((e = cudaMemcpy(word, status, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess)
      return cuda_fail(e, "cudaMemcpy(status)");
    if (word[0] != 0 && (e = cudaMemset(status, 0, sizeof(word))) != cudaSuccess)
      return cuda_fail(e, "cudaMemset(status)");
  }
  uint32_t word2[4] = {0, 0, 0, 0};
  int rc = noalloc_take_status(dev, word2);
  if (rc != ATTN_OK) return rc;
  if (word[0] == 0) std::memcpy(word, word2, sizeof(word));
  if (detail) std::memcpy(detail, word, sizeof(word));
  if (word[0] == 0) return ATTN_OK;
  if (word[0] == ATTN_ERR_TIMEOUT)
    return fail(ATTN_ERR_TIMEOUT, "device wait ran out: role %u, KV tile %d, CTA %u", word[1],
                static_cast<int>(word[2]), word[3]);
  return fail(ATTN_ERR_CUDA, "unexpected device status %u", word[0]);
}

const char* attn_error_string(int code) {
  switch (code) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "misaligned pointer or stride";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status code";
  }
}

const char* attn_last_error(void) { return t_err; }

int attn_device_sm_count(void) {
  DeviceState* ds = nullptr;
  int rc = device_state(&ds);
  if (rc != ATTN_OK) return -rc;
  return ds->sm_count;
}

int attn_tune(const attn_params_ex* p, int iters, attn_tune_result* out) {
  t_err[0] = 0;
  if (!p || !out) return fail(ATTN_ERR_INVALID_ARG, "params and result must be non-null");
  if (iters < 1) return fail(ATTN_ERR_INVALID_ARG, "iters must be >= 1");
  DeviceState* ds = nullptr;
  int rc;
  if ((rc = device_state(&ds)) != ATTN_OK) return rc;
  const int sm = ds->sm_count;
  // candidates: (schedule, num_ctas)
  int cand[16][2];
  int nc = 0;
  cand[nc][0] = 1;
  cand[nc][1] = 0;
  ++nc;
  if (p->mask_kind == ATTN_MASK_NONE) {
    const int fr[] = {8, 7, 6, 5, 4, 3, 2};  // G = sm * fr / 8
    for (int f : fr) {
      const int g = sm * f / 8;
      if (g < 1 || g > attn::kMaxSplitCtas) continue;
      bool dup = false;
      for (int i = 0; i < nc; ++i) dup |= cand[i][0] == 2 && cand[i][1] == g;
      if (dup) continue;
      cand[nc][0] = 2;
      cand[nc][1] = g;
      ++nc;
    }
  }
  cudaStream_t s = p->stream ? static_cast<cudaStream_t>(p->stream) : t_stream;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  cudaError_t e;
  if ((e = cudaEventCreate(&e0)) != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
  if ((e = cudaEventCreate(&e1)) != cudaSuccess) {
    cudaEventDestroy(e0);
    return cuda_fail(e, "cudaEventCreate");
  }
  float best = 0.f;
  int best_i = -1;
  rc = ATTN_OK;
  for (int i = 0; i < nc && rc == ATTN_OK; ++i) {
    attn_params_ex c = *p;
    c.schedule = cand[i][0];
    c.num_ctas = cand[i][1];
    c.ev_start = c.ev_stop = nullptr;
    // two untimed launches (workspace growth, caches), then `iters` timed ones
    for (int w = 0; w < 2 && rc == ATTN_OK; ++w) rc = attn_fwd_ex(&c);
    if (rc != ATTN_OK) break;
    if ((e = cudaEventRecord(e0, s)) != cudaSuccess) { rc = cuda_fail(e, "cudaEventRecord"); break; }
    for (int it = 0; it < iters && rc == ATTN_OK; ++it) rc = attn_fwd_ex(&c);
    if (rc != ATTN_OK) break;
    if ((e = cudaEventRecord(e1, s)) != cudaSuccess) { rc = cuda_fail(e, "cudaEventRecord"); break; }
    if ((e = cudaEventSynchronize(e1)) != cudaSuccess) { rc = cuda_fail(e, "cudaEventSynchronize"); break; }
    float ms = 0.f;
    if ((e = cudaEventElapsedTime(&ms, e0, e1)) != cudaSuccess) { rc = cuda_fail(e, "cudaEventElapsedTime"); break; }
    const float us = 1000.f * ms / static_cast<float>(iters);
    if (best_i < 0 || us < best) {
      best = us;
      best_i = i;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (rc != ATTN_OK) return rc;
  out->schedule = cand[best_i][0];
  out->num_ctas = cand[best_i][1];
  out->us = best;
  out->n_tried = nc;
  return ATTN_OK;
}

void attn_shutdown(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  noalloc_forget();  // the next no-alloc call looks the array's address up again
  for (int i = 0; i < kMaxDevices; ++i) {
    if (g_dev[i].status) {
      int prev = 0;
      cudaGetDevice(&prev);
      if (cudaSetDevice(i) == cudaSuccess) {
        cudaFree(g_dev[i].status);
        if (g_dev[i].ws) cudaFree(g_dev[i].ws);
        if (g_dev[i].dd) cudaFree(g_dev[i].dd);
        if (g_dev[i].aux) cudaStreamDestroy(g_dev[i].aux);
        if (g_dev[i].fork) cudaEventDestroy(g_dev[i].fork);
        if (g_dev[i].join) cudaEventDestroy(g_dev[i].join);
      }
      cudaSetDevice(prev);
      g_dev[i].status = nullptr;
      g_dev[i].ws = nullptr;
      g_dev[i].ws_bytes = 0;
      g_dev[i].dd = nullptr;
      g_dev[i].dd_bytes = 0;
      g_dev[i].aux = nullptr;
      g_dev[i].fork = g_dev[i].join = nullptr;
    }
  }
}

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

int64_t attn_workspace_bytes(const attn_params_ex* p) {
  t_err[0] = 0;
  Checked c;
  int rc = validate(p, &c);
  if (rc != ATTN_OK) return -rc;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != ATTN_OK) return -rc;
  Plan pl;
  if ((rc = make_plan(p, ds->sm_count, &pl)) != ATTN_OK) return -rc;
  return static_cast<int64_t>(pl.ws_bytes());
}

int attn_params_size(void) { return static_cast<int>(sizeof(attn_params_ex)); }

void attn_bwd_params_init(attn_bwd_params* p) {
  if (!p) return;
  std::memset(p, 0, sizeof(*p));
  p->dilation = 1;
}

int attn_bwd(const attn_bwd_params* p) {
  t_err[0] = 0;
  if (!p) return fail(ATTN_ERR_INVALID_ARG, "params is NULL");
  // the forward's checks, on the forward's view of the problem
  attn_params_ex fp;
  attn_params_init(&fp);
  fp.q = p->q;
  fp.k = p->k;
  fp.v = p->v;
  fp.o = const_cast<void*>(p->o);
  fp.lse = const_cast<float*>(p->lse);
  fp.B = p->B;
  fp.H = p->H;
  fp.Nq = p->Nq;
  fp.Nk = p->Nk;
  fp.d = p->d;
  fp.scale = p->scale;
  fp.mask_kind = p->mask_kind;
  fp.window = p->window;
  fp.window_w = p->window_w;
  fp.dilation = p->dilation;
  fp.wrap = p->wrap;
  fp.grid_h = p->grid_h;
  fp.grid_w = p->grid_w;
  fp.grid_d = p->grid_d;
  fp.window_d = p->window_d;
  fp.wrap_d = p->wrap_d;
  Checked c;
  int rc = validate(&fp, &c);
  if (rc != ATTN_OK) return rc;
  const int64_t BH = static_cast<int64_t>(p->B) * p->H;
  if (BH * ((p->Nq + 127) / 128) >= (int64_t{1} << 31) || BH * ((p->Nk + 127) / 128) >= (int64_t{1} << 31))
    return fail(ATTN_ERR_INVALID_ARG, "too many tiles");
  const void* ptrs[] = {p->dout, p->lse, p->dq, p->dk, p->dv};
  for (const void* x : ptrs) {
    if (!x) return fail(ATTN_ERR_INVALID_ARG, "dout, lse, dq, dk, dv must be non-null");
    if (!aligned16(x)) return fail(ATTN_ERR_MISALIGNED, "every pointer must be 16-byte aligned");
  }
  if ((rc = get_encoder()) != ATTN_OK) return rc;
  DeviceState* ds = nullptr;
  if ((rc = device_state(&ds)) != ATTN_OK) return rc;
  const size_t need = static_cast<size_t>(BH) * p->Nq * sizeof(float);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (ds->dd_bytes < need) {
      cudaError_t e;
      if (ds->dd) {
        if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(ds->dd);
        ds->dd = nullptr;
        ds->dd_bytes = 0;
      }
      void* ptr = nullptr;
      if ((e = cudaMalloc(&ptr, need)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(backward scratch)");
      ds->dd = static_cast<float*>(ptr);
      ds->dd_bytes = need;
    }
    if (!ds->aux) {
      cudaError_t e;
      if ((e = cudaStreamCreateWithFlags(&ds->aux, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_fail(e, "cudaStreamCreateWithFlags");
      if ((e = cudaEventCreateWithFlags(&ds->fork, cudaEventDisableTiming)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&ds->join, cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e, "cudaEventCreateWithFlags");
    }
  }
  attn::BwdParams bp;
  std::memset(&bp, 0, sizeof(bp));
  attn::KernelParams& kp = bp.f;
  const int box_cols = p->d >= 64 ? 64 : 32;
  const CUtensorMapSwizzle swz = p->d >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  const int64_t qs[3] = {static_cast<int64_t>(p->H) * p->Nq * p->d, static_cast<int64_t>(p->Nq) * p->d, p->d};
  const int64_t ks[3] = {static_cast<int64_t>(p->H) * p->Nk * p->d, static_cast<int64_t>(p->Nk) * p->d, p->d};
  if ((rc = encode_map(&kp.tm_q, p->q, p->d, p->Nq, p->H, p->B, qs, box_cols, swz, "q")) != ATTN_OK ||
      (rc = encode_map(&kp.tm_k, p->k, p->d, p->Nk, p->H, p->B, ks, box_cols, swz, "k")) != ATTN_OK ||
      (rc = encode_map(&kp.tm_v, p->v, p->d, p->Nk, p->H, p->B, ks, box_cols, swz, "v")) != ATTN_OK ||
      (rc = encode_map(&bp.tm_do, p->dout, p->d, p->Nq, p->H, p->B, qs, box_cols, swz, "dout")) != ATTN_OK)
    return rc;
  kp.B = p->B;
  kp.H = p->H;
  kp.Nq = p->Nq;
  kp.Nk = p->Nk;
  kp.c = p->scale * 1.4426950408889634f;
  const int mask = kernel_mask(&fp, c, &kp);
  kp.n_kv = (p->Nk + attn::kBN - 1) / attn::kBN;
  kp.timeout_ns = p->timeout_ns ? p->timeout_ns : kDefaultTimeoutNs;
  kp.status = ds->status;
  bp.o = p->o;
  bp.dout = p->dout;
  bp.lse = p->lse;
  bp.dd = ds->dd;
  bp.dq = p->dq;
  bp.dk = p->dk;
  bp.dv = p->dv;
  bp.scale = p->scale;
  cudaStream_t s = p->stream ? static_cast<cudaStream_t>(p->stream) : t_stream;
  const cudaError_t e = attn::launch_bwd(bp, p->d, mask, s, ds->aux, ds->fork, ds->join);
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return ATTN_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- no-alloc entry point
//
// attn_fwd_noalloc: for callers that cannot allocate device memory at all --
// code running where cudaMalloc is forbidden or unavailable (inside a memory
// pool's own bookkeeping, a custom allocator, an embedded runtime that owns
// every allocation), or that must not allocate lazily on a first call. It
// runs the split-schedule unmasked forward pass with all of its scratch (the
// partial results of cut tasks, their arrival words and the device status
// word) in one fixed, file-scope device array, so it calls no cudaMalloc,
// cudaFree or other allocating routine.
namespace {

// Fixed scratch of the no-alloc entry point. Every GPU on which the library's
// device code is loaded holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t{48} << 20;
constexpr size_t kNoAllocStatusBytes = 256;  // device status word at the front
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sm_count = 0;
  uint32_t epoch = 0;                // tag of the last call on this device (never reset: the
                                     // array keeps earlier calls' arrival words)
};
NoAllocDevice g_noalloc[kMaxDevices];

// Once per device (again after attn_shutdown), with that device current: the
// device address of the scratch array (the symbol name itself is only a
// host-side stand-in).
int noalloc_setup(NoAllocDevice** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (d.scratch == nullptr) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (major != 10 || minor != 3)
      return fail(ATTN_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                  dev, major, minor);
    void* ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    d.sm_count = sms;
    d.scratch = static_cast<unsigned char*>(ptr);
  }
  *out = &d;
  return ATTN_OK;
}

int noalloc_take_status(int dev, uint32_t word[4]) {
  word[0] = word[1] = word[2] = word[3] = 0;
  bool used;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    used = g_noalloc[dev].scratch != nullptr;
  }
  if (!used) return ATTN_OK;
  cudaError_t e = cudaMemcpyFromSymbol(word, g_noalloc_scratch, 4 * sizeof(uint32_t), 0,
                                       cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol(no-alloc status)");
  if (word[0] != 0) {
    const uint32_t zero[4] = {0, 0, 0, 0};
    if ((e = cudaMemcpyToSymbol(g_noalloc_scratch, zero, sizeof(zero), 0,
                                cudaMemcpyHostToDevice)) != cudaSuccess)
      return cuda_fail(e, "cudaMemcpyToSymbol(no-alloc status)");
  }
  return ATTN_OK;
}

void noalloc_forget() {
  for (int i = 0; i < kMaxDevices; ++i) g_noalloc[i].scratch = nullptr;
}

}  // namespace

extern "C" int attn_fwd_noalloc(const attn_params_ex* p) {
  t_err[0] = 0;
  Checked c;
  int rc = validate(p, &c);
  if (rc != ATTN_OK) return rc;
  if (p->mask_kind != ATTN_MASK_NONE)
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_noalloc computes unmasked attention only");
  if (p->workspace != nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_noalloc uses its own fixed scratch; workspace must be NULL");
  if ((rc = get_encoder()) != ATTN_OK) return rc;
  NoAllocDevice* nd = nullptr;
  if ((rc = noalloc_setup(&nd)) != ATTN_OK) return rc;

  attn_params_ex split = *p;
  split.schedule = 2;
  Plan pl;
  if ((rc = make_plan(&split, nd->sm_count, &pl)) != ATTN_OK) return rc;
  const size_t need = kNoAllocStatusBytes + pl.ws_bytes();
  if (need > kNoAllocScratchBytes)
    return fail(ATTN_ERR_INVALID_ARG,
                "this problem needs %zu bytes of scratch; attn_fwd_noalloc has %zu (use attn_fwd_ex)",
                need, kNoAllocScratchBytes);

  attn::KernelParams kp;
  int mask = 0;
  if ((rc = fill_params(&split, c, pl, &kp, &mask)) != ATTN_OK) return rc;
  // Layout of the scratch: status word, partial results, arrival words. The
  // arrival words carry each call's tag, so nothing has to be cleared between
  // calls (the array starts zeroed, and tag 0 is never used).
  kp.status = reinterpret_cast<uint32_t*>(nd->scratch);
  if (pl.split) {
    kp.ws_part = reinterpret_cast<float*>(nd->scratch + kNoAllocStatusBytes);
    kp.ws_count = reinterpret_cast<unsigned long long*>(nd->scratch + kNoAllocStatusBytes +
                                                         align256(pl.part_bytes));
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (++nd->epoch == 0) nd->epoch = 1;
    kp.epoch = nd->epoch;
  }
  log_launch("attn_fwd_noalloc", p, kp, mask, pl);
  cudaStream_t s = p->stream ? static_cast<cudaStream_t>(p->stream) : t_stream;
  cudaError_t e;
  if (p->ev_start && (e = cudaEventRecord(static_cast<cudaEvent_t>(p->ev_start), s)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord(start)");
  switch (p->d) {
    case 32: e = attn::launch_d32(kp, mask, pl.grid, s); break;
    case 64: e = attn::launch_d64(kp, mask, pl.grid, s); break;
    default: e = attn::launch_d128(kp, mask, pl.grid, s); break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  if (p->ev_stop && (e = cudaEventRecord(static_cast<cudaEvent_t>(p->ev_stop), s)) != cudaSuccess)
    return cuda_fail(e, "cudaEventRecord(stop)");
  return ATTN_OK;
}
