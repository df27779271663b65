// Host build of the kernel's tile planning (which K/V tiles a Q tile visits,
// and which of them need the in-tile mask), for CPU tests against the oracle.
#include "attn_sm103.cuh"

namespace {
template <int MASK>
int cls(int q0, int j, const attn::KernelParams& p) { return attn::dev::tile_class<MASK>(q0, j, p); }
}

extern "C" int tile_class_host(int mask, int q0, int j, int Nq, int Nk, int grid_h, int grid_w,
                               int window, int dilation) {
  attn::KernelParams p{};
  p.Nq = Nq;
  p.Nk = Nk;
  p.grid_h = grid_h;
  p.grid_w = grid_w;
  p.window = window;
  p.dilation = dilation;
  p.n_kv = (Nk + attn::kBN - 1) / attn::kBN;
  const bool dil = dilation > 1;
  switch (mask) {
    case attn::kMaskNone: return cls<attn::kMaskNone>(q0, j, p);
    case attn::kMaskCausal: return cls<attn::kMaskCausal>(q0, j, p);
    case attn::kMaskNaClamp:
      return dil ? cls<attn::kMaskNaClampDil>(q0, j, p) : cls<attn::kMaskNaClamp>(q0, j, p);
    case attn::kMaskNaWrap:
      return dil ? cls<attn::kMaskNaWrapDil>(q0, j, p) : cls<attn::kMaskNaWrap>(q0, j, p);
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
extern "C" void na_bits_host(int wrap, int q, int k0, int N, int grid_h, int grid_w, int window,
                             int dilation, unsigned* out) {
  attn::KernelParams p{};
  p.Nq = p.Nk = N;
  p.grid_h = grid_h;
  p.grid_w = grid_w;
  p.window = window;
  p.dilation = dilation;
  int qy, qx, wy, wx;
  uint32_t bits[4];
  const bool dil = dilation > 1;
  if (wrap && dil) {
    attn::dev::na_query_coords<true, true>(p, q, qy, qx, wy, wx);
    attn::dev::na_tile_bits<true, true>(p, k0, qy, qx, wy, wx, bits);
  } else if (wrap) {
    attn::dev::na_query_coords<true, false>(p, q, qy, qx, wy, wx);
    attn::dev::na_tile_bits<true, false>(p, k0, qy, qx, wy, wx, bits);
  } else if (dil) {
    attn::dev::na_query_coords<false, true>(p, q, qy, qx, wy, wx);
    attn::dev::na_tile_bits<false, true>(p, k0, qy, qx, wy, wx, bits);
  } else {
    attn::dev::na_query_coords<false, false>(p, q, qy, qx, wy, wx);
    attn::dev::na_tile_bits<false, false>(p, k0, qy, qx, wy, wx, bits);
  }
  for (int i = 0; i < 4; ++i) out[i] = bits[i];
}
