// Host build of the kernel's tile planning (which K/V tiles a Q tile visits,
// and which of them need the in-tile mask), for CPU tests against the oracle.
#include "attn_sm103.cuh"

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

// Task index -> (b, h, first row of Q tile 0), as the kernel decodes it.
extern "C" void decode_task_host(int mask, int t, int B, int H, int Nq, int* out) {
  attn::KernelParams p{};
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.n_qpairs = (Nq + 2 * attn::kBM - 1) / (2 * attn::kBM);
  attn::dev::Task k = mask == attn::kMaskCausal ? attn::dev::decode_task<attn::kMaskCausal>(t, p)
                                                : attn::dev::decode_task<attn::kMaskNone>(t, p);
  out[0] = k.b;
  out[1] = k.h;
  out[2] = k.q0[0];
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
