// Host build of the kernel's tile planning (which K/V tiles a Q tile visits,
// and which of them need the in-tile mask), for CPU tests against the oracle.
#include "attn_sm103.cuh"
#include "attn_bwd_sm103.cuh"

namespace {
template <int MASK>
int cls(int q0, int j, const attn::KernelParams& p) { return attn::dev::tile_class<MASK>(q0, j, p); }

template <int MASK>
void bits_of(const attn::KernelParams& p, int q, int k0, uint32_t (&bits)[4]) {
  constexpr bool WH = attn::mask_na_wrap_rows(MASK), WW = attn::mask_na_wrap_cols(MASK);
  constexpr bool DIL = attn::mask_na_dilated(MASK);
  int qy, qx, wy, wx;
  attn::dev::na_query_coords<WH, WW, DIL>(p, q, qy, qx, wy, wx);
  attn::dev::na_tile_bits<WH, WW, DIL>(p, k0, qy, qx, wy, wx, bits);
}

attn::KernelParams na_params(int Nq, int Nk, int grid_h, int grid_w, int window_h, int window_w,
                             int dilation) {
  attn::KernelParams p{};
  p.Nq = Nq;
  p.Nk = Nk;
  p.grid_h = grid_h;
  p.grid_w = grid_w;
  p.window_h = window_h;
  p.window_w = window_w;
  p.dilation = dilation;
  p.n_kv = (Nk + attn::kBN - 1) / attn::kBN;
  return p;
}
}  // namespace

// kind: 0 no mask, 1 causal, 2 neighbourhood (with the per-axis options).
extern "C" int tile_class_host(int kind, int q0, int j, int Nq, int Nk, int grid_h, int grid_w,
                               int window_h, int window_w, int dilation, int wrap_rows,
                               int wrap_cols) {
  const attn::KernelParams p = na_params(Nq, Nk, grid_h, grid_w, window_h, window_w, dilation);
  if (kind == 0) return cls<attn::kMaskNone>(q0, j, p);
  if (kind == 1) return cls<attn::kMaskCausal>(q0, j, p);
  if (kind != 2) return -1;
  switch (attn::na_mask(wrap_rows != 0, wrap_cols != 0, dilation > 1)) {
    case attn::kMaskNa + 0: return cls<attn::kMaskNa + 0>(q0, j, p);
    case attn::kMaskNa + 1: return cls<attn::kMaskNa + 1>(q0, j, p);
    case attn::kMaskNa + 2: return cls<attn::kMaskNa + 2>(q0, j, p);
    case attn::kMaskNa + 3: return cls<attn::kMaskNa + 3>(q0, j, p);
    case attn::kMaskNa + 4: return cls<attn::kMaskNa + 4>(q0, j, p);
    case attn::kMaskNa + 5: return cls<attn::kMaskNa + 5>(q0, j, p);
    case attn::kMaskNa + 6: return cls<attn::kMaskNa + 6>(q0, j, p);
    case attn::kMaskNa + 7: return cls<attn::kMaskNa + 7>(q0, j, p);
    default: return -1;
  }
}

// Task index -> (b, h, first row of Q tile 0, whether Q tile 1 is live), as
// the kernel decodes it with q_tiles Q tiles per task.
extern "C" void decode_task_host(int mask, int t, int B, int H, int Nq, int q_tiles, int* out) {
  attn::KernelParams p{};
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.q_tiles = q_tiles;
  p.n_qtasks = (Nq + q_tiles * attn::kBM - 1) / (q_tiles * attn::kBM);
  attn::dev::Task k = mask == attn::kMaskCausal ? attn::dev::decode_task<attn::kMaskCausal>(t, p)
                                                : attn::dev::decode_task<attn::kMaskNone>(t, p);
  out[0] = k.b;
  out[1] = k.h;
  out[2] = k.q0[0];
  out[3] = k.live[1] ? 1 : 0;
}

// The in-tile neighbourhood mask of query q for the K/V tile starting at key
// k0: bit i set iff key k0 + i is allowed.
extern "C" void na_bits_host(int q, int k0, int N, int grid_h, int grid_w, int window_h,
                             int window_w, int dilation, int wrap_rows, int wrap_cols,
                             unsigned* out) {
  const attn::KernelParams p = na_params(N, N, grid_h, grid_w, window_h, window_w, dilation);
  uint32_t bits[4] = {0u, 0u, 0u, 0u};
  switch (attn::na_mask(wrap_rows != 0, wrap_cols != 0, dilation > 1)) {
    case attn::kMaskNa + 0: bits_of<attn::kMaskNa + 0>(p, q, k0, bits); break;
    case attn::kMaskNa + 1: bits_of<attn::kMaskNa + 1>(p, q, k0, bits); break;
    case attn::kMaskNa + 2: bits_of<attn::kMaskNa + 2>(p, q, k0, bits); break;
    case attn::kMaskNa + 3: bits_of<attn::kMaskNa + 3>(p, q, k0, bits); break;
    case attn::kMaskNa + 4: bits_of<attn::kMaskNa + 4>(p, q, k0, bits); break;
    case attn::kMaskNa + 5: bits_of<attn::kMaskNa + 5>(p, q, k0, bits); break;
    case attn::kMaskNa + 6: bits_of<attn::kMaskNa + 6>(p, q, k0, bits); break;
    case attn::kMaskNa + 7: bits_of<attn::kMaskNa + 7>(p, q, k0, bits); break;
    default: break;
  }
  for (int i = 0; i < 4; ++i) out[i] = bits[i];
}

namespace {
attn::KernelParams na3_params(int N, int grid_d, int grid_h, int grid_w, int window_d, int window_h,
                              int window_w, int dilation, int wrap_bits) {
  attn::KernelParams p = na_params(N, N, grid_h, grid_w, window_h, window_w, dilation);
  p.grid_d = grid_d;
  p.window_d = window_d;
  p.na_wrap = wrap_bits;
  return p;
}

int na2_mask(int wrap_rows, int wrap_cols, int dilation) {
  return attn::na_mask(wrap_rows != 0, wrap_cols != 0, dilation > 1);
}

template <int MASK>
void key_bits_of(const attn::KernelParams& p, int q0, int kk, uint32_t (&bits)[4]) {
  attn::dev::na_key_bits<MASK>(p, q0, kk, bits);
}
}  // namespace

// Volumes: wrap_bits 1 columns, 2 rows, 4 depth.
extern "C" int tile_class3_host(int q0, int j, int N, int grid_d, int grid_h, int grid_w,
                                int window_d, int window_h, int window_w, int dilation,
                                int wrap_bits) {
  const attn::KernelParams p =
      na3_params(N, grid_d, grid_h, grid_w, window_d, window_h, window_w, dilation, wrap_bits);
  return cls<attn::kMaskNa3>(q0, j, p);
}

extern "C" void na3_bits_host(int q, int k0, int N, int grid_d, int grid_h, int grid_w,
                              int window_d, int window_h, int window_w, int dilation,
                              int wrap_bits, unsigned* out) {
  const attn::KernelParams p =
      na3_params(N, grid_d, grid_h, grid_w, window_d, window_h, window_w, dilation, wrap_bits);
  uint32_t bits[4];
  attn::dev::na3_tile_bits(p, k0, attn::dev::na_query<attn::kMaskNa3>(p, q), bits);
  for (int i = 0; i < 4; ++i) out[i] = bits[i];
}

// The backward's transposed mask: bit e set iff query q0 + e has key kk in its
// window. grid_d == 0: a 2-D grid (wrap_bits 1 columns, 2 rows); else a volume.
extern "C" void na_key_bits_host(int q0, int kk, int N, int grid_d, int grid_h, int grid_w,
                                 int window_d, int window_h, int window_w, int dilation,
                                 int wrap_bits, unsigned* out) {
  const attn::KernelParams p =
      na3_params(N, grid_d, grid_h, grid_w, window_d, window_h, window_w, dilation, wrap_bits);
  uint32_t bits[4] = {0u, 0u, 0u, 0u};
  if (grid_d > 0) {
    key_bits_of<attn::kMaskNa3>(p, q0, kk, bits);
  } else {
    switch (na2_mask(wrap_bits & 2, wrap_bits & 1, dilation)) {
      case attn::kMaskNa + 0: key_bits_of<attn::kMaskNa + 0>(p, q0, kk, bits); break;
      case attn::kMaskNa + 1: key_bits_of<attn::kMaskNa + 1>(p, q0, kk, bits); break;
      case attn::kMaskNa + 2: key_bits_of<attn::kMaskNa + 2>(p, q0, kk, bits); break;
      case attn::kMaskNa + 3: key_bits_of<attn::kMaskNa + 3>(p, q0, kk, bits); break;
      case attn::kMaskNa + 4: key_bits_of<attn::kMaskNa + 4>(p, q0, kk, bits); break;
      case attn::kMaskNa + 5: key_bits_of<attn::kMaskNa + 5>(p, q0, kk, bits); break;
      case attn::kMaskNa + 6: key_bits_of<attn::kMaskNa + 6>(p, q0, kk, bits); break;
      case attn::kMaskNa + 7: key_bits_of<attn::kMaskNa + 7>(p, q0, kk, bits); break;
      default: break;
    }
  }
  for (int i = 0; i < 4; ++i) out[i] = bits[i];
}

// The band of candidate tiles for the 128-token tile starting at t0: out =
// {lo0, hi0, lo1, hi1}. grid_d == 0: a 2-D grid (wrap_bits 1 columns, 2 rows).
extern "C" void band_host(int t0, int N, int grid_d, int grid_h, int grid_w, int window_d,
                          int window_h, int window_w, int dilation, int wrap_bits, int* out) {
  const attn::KernelParams p =
      na3_params(N, grid_d, grid_h, grid_w, window_d, window_h, window_w, dilation, wrap_bits);
  const int t1 = (t0 + attn::kBM < N ? t0 + attn::kBM : N) - 1;
  attn::dev::Band b{};
  if (grid_d > 0) {
    b = attn::dev::na_band<attn::kMaskNa3>(t0, t1, p);
  } else {
    switch (na2_mask(wrap_bits & 2, wrap_bits & 1, dilation)) {
      case attn::kMaskNa + 0: b = attn::dev::na_band<attn::kMaskNa + 0>(t0, t1, p); break;
      case attn::kMaskNa + 1: b = attn::dev::na_band<attn::kMaskNa + 1>(t0, t1, p); break;
      case attn::kMaskNa + 2: b = attn::dev::na_band<attn::kMaskNa + 2>(t0, t1, p); break;
      case attn::kMaskNa + 3: b = attn::dev::na_band<attn::kMaskNa + 3>(t0, t1, p); break;
      case attn::kMaskNa + 4: b = attn::dev::na_band<attn::kMaskNa + 4>(t0, t1, p); break;
      case attn::kMaskNa + 5: b = attn::dev::na_band<attn::kMaskNa + 5>(t0, t1, p); break;
      case attn::kMaskNa + 6: b = attn::dev::na_band<attn::kMaskNa + 6>(t0, t1, p); break;
      case attn::kMaskNa + 7: b = attn::dev::na_band<attn::kMaskNa + 7>(t0, t1, p); break;
      default: break;
    }
  }
  out[0] = b.lo0;
  out[1] = b.hi0;
  out[2] = b.lo1;
  out[3] = b.hi1;
}

// Whether a launch with one Q tile per task (fewer Q-tile pairs than CTAs)
// runs its tasks as twins: the decision the host takes at launch. grid_d == 0:
// a 2-D grid (wrap_bits 1 columns, 2 rows); else a volume (4 depth as well).
extern "C" int twin_host(int B, int H, int N, int grid_d, int grid_h, int grid_w, int window_d,
                         int window_h, int window_w, int dilation, int wrap_bits) {
  attn::KernelParams p =
      na3_params(N, grid_d, grid_h, grid_w, window_d, window_h, window_w, dilation, wrap_bits);
  p.B = B;
  p.H = H;
  p.q_tiles = 1;
  p.n_qtasks = (N + attn::kBM - 1) / attn::kBM;
  p.n_tasks = B * H * p.n_qtasks;
  const int mask = grid_d == 0 ? na2_mask(wrap_bits & 2, wrap_bits & 1, dilation) : attn::kMaskNa3;
  return attn::dev::twin_dim(p, mask);
}
