// attn_bwd_sm103.cuh -- backward pass of the fused exact attention on sm_103a:
// dQ, dK, dV from Q, K, V, O, dO and the forward's log-sum-exp.
//
// With P = exp(scale Q K^T - LSE) (row softmax, recomputed from the saved LSE)
// and D_i = dO_i . O_i:
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D),   dQ = scale dS K,
//   dK = scale dS^T Q
// (the chain rule through S = Q K^T, the row softmax and R = S V, "Fused Self
// Attention", section "Background").
//
// Three kernels. The first computes D. The second keeps one 128-row Q tile
// (and its dO) in shared memory and streams the K/V tiles it attends: S and dP
// by tcgen05.mma into TMEM, P and dS by one thread per query row, dQ += dS K
// with dS (bf16) from TMEM. The third keeps one 128-key K/V tile and streams
// the Q/dO tiles that attend it: S^T = K Q^T and dP^T = V dO^T (keys on the
// TMEM lanes), P^T and dS^T by one thread per key row, dV += P^T dO and
// dK += dS^T Q with the A operand from TMEM. Every product uses the operand
// forms of the forward kernel: K-major A and B from shared memory, A from
// TMEM, MN-major B from shared memory.
#pragma once

#include "attn_sm103.cuh"

namespace attn {
namespace dev {

constexpr int kBwdThreads = 256;  // warp 0 loader, warp 1 MMA issuer, warps 4-7 one row each

template <int D>
struct BwdCfg {
  using C = Cfg<D>;
  static constexpr int kStages = D == 128 ? 2 : (D == 64 ? 3 : 4);
  // stationary pair (Q, dO or K, V), then a ring of the streamed pairs
  static constexpr int kOffA = 0;
  static constexpr int kOffB = C::kTileBytes;
  static constexpr int kOffRing = 2 * C::kTileBytes;
  static constexpr int kRingStride = 2 * C::kTileBytes;
  static constexpr int kOffVec = kOffRing + kStages * kRingStride;   // per stage: lse2[128], d[128]
  static constexpr int kVecBytes = 2 * 128 * 4;
  static constexpr int kOffBar = kOffVec + kStages * kVecBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static constexpr uint32_t kIdescNN = make_idesc(kBM, kBN, false);  // S, dP: N = 128 keys / rows
  static constexpr uint32_t kIdescMN = make_idesc(kBM, D, true);     // dQ, dK, dV: N = d
};

// Barrier slots of the backward kernels.
struct BwdBars {
  uint32_t base;
  int st;
  __device__ uint32_t a_full() const { return base; }              // stationary pair landed
  __device__ uint32_t s_full() const { return base + 8; }          // S (or S^T) and dP ready
  __device__ uint32_t g_full() const { return base + 16; }         // dS (and P) in TMEM
  __device__ uint32_t acc_full() const { return base + 24; }       // accumulators final
  __device__ uint32_t done() const { return base + 32; }
  __device__ uint32_t ring_full(int s) const { return base + 40 + 8 * s; }
  __device__ uint32_t ring_empty(int s) const { return base + 40 + 8 * (st + s); }
  __device__ int count() const { return 5 + 2 * st; }
};

// D_i = sum_t dO_it O_it (fp32), one thread per row; rows contiguous, d bf16 each.
__global__ void bwd_rowdot_kernel(const __nv_bfloat16* __restrict__ o,
                                  const __nv_bfloat16* __restrict__ dout, float* __restrict__ dd,
                                  int64_t rows, int d) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  const uint4* a = reinterpret_cast<const uint4*>(o + r * d);
  const uint4* b = reinterpret_cast<const uint4*>(dout + r * d);
  float acc = 0.f;
  for (int i = 0; i < d / 8; ++i) {
    const uint4 x = a[i], y = b[i];
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[t]));
      const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[t]));
      acc = fmaf(fx.x, fy.x, acc);
      acc = fmaf(fx.y, fy.y, acc);
    }
  }
  dd[r] = acc;
}

// D (tmem) = A (smem, K-major, 128 rows) B^T (smem, K-major, 128 rows), K = d.
template <int D>
__device__ __forceinline__ void issue_nn(uint32_t d_tmem, uint32_t a_tile, uint32_t b_tile) {
  using C = Cfg<D>;
  a_tile = opaque(a_tile);
  b_tile = opaque(b_tile);
  const uint64_t a0 = smem_desc(a_tile, 16, 8 * C::kSwizzle, C::kLayout);
  const uint64_t b0 = smem_desc(b_tile, 16, 8 * C::kSwizzle, C::kLayout);
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t off = ((ks * 16) / C::kBoxCols) * C::kChunkBytes + ((ks * 16) % C::kBoxCols) * 2;
    mma_ss(d_tmem, a0 + (off >> 4), b0 + (off >> 4), BwdCfg<D>::kIdescNN, ks > 0 ? 1u : 0u);
  }
}

// D (tmem, 128 x d) (+)= A (tmem, bf16 128 x 128) B (smem, 128 rows x d, MN-major).
template <int D>
__device__ __forceinline__ void issue_tmn(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_tile,
                                          bool accumulate) {
  using C = Cfg<D>;
  b_tile = opaque(b_tile);
  const uint64_t b0 = smem_desc(b_tile, C::kChunkBytes, 8 * C::kSwizzle, C::kLayout);
#pragma unroll
  for (int ks = 0; ks < kBN / 16; ++ks)
    mma_ts(d_tmem, a_tmem + ks * 8, b0 + ((ks * 16 * C::kSwizzle) >> 4), BwdCfg<D>::kIdescMN,
           (accumulate || ks > 0) ? 1u : 0u);
}

template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* m, uint32_t bar, int row,
                                          int h, int b) {
  using C = Cfg<D>;
  for (int c = 0; c < C::kChunks; ++c)
    tma_load_4d(dst + c * C::kChunkBytes, m, bar, c * C::kBoxCols, row, h, b);
}

// Stores 32 bf16 pairs from a thread's row (packed) into consecutive TMEM columns.
__device__ __forceinline__ void store_packed32(uint32_t taddr, const uint32_t (&pk)[32]) {
  tmem_st32(taddr, pk);
}

// Tiles of the other side a 128-token tile starting at t0 (of n tokens) may
// meet: the neighbourhood band, else all `tiles`.
template <int MASK>
__host__ __device__ __forceinline__ Band bwd_band(int t0, int n, int tiles, const KernelParams& p) {
  if constexpr (mask_is_na(MASK)) {
    return na_band<MASK>(t0, min(t0 + kBM, n) - 1, p);
  } else {
    Band b;
    b.lo0 = 0;
    b.hi0 = tiles;
    b.lo1 = b.hi1 = 0;
    return b;
  }
}

// ------------------------------------------------------------------ dQ

// One CTA per (batch, head, 128-row Q tile).
template <int D, int MASK>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdParams bp) {
  using C = Cfg<D>;
  using BC = BwdCfg<D>;
  const KernelParams& p = bp.f;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BwdBars bars{sbase + BC::kOffBar, BC::kStages};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + BC::kOffBar + 8 * bars.count());
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const int n_qt = (p.Nq + kBM - 1) / kBM;
  const int bh = blockIdx.x / n_qt;
  const int q0 = (blockIdx.x - bh * n_qt) * kBM;
  const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
  const Band band = bwd_band<MASK>(q0, p.Nq, p.n_kv, p);  // K/V tiles this Q tile may meet

  if (threadIdx.x == 0) {
    mbar_init(bars.a_full(), 1);
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.g_full(), 4);
    mbar_init(bars.acc_full(), 1);
    mbar_init(bars.done(), 1);
    for (int s = 0; s < BC::kStages; ++s) {
      mbar_init(bars.ring_full(s), 1);
      mbar_init(bars.ring_empty(s), 1);
    }
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    // Q and dO of this tile, then K and V of every tile it attends
    int armed_a = -1, armed[4] = {-1, -1, -1, -1};
    uint32_t it = 0;
    mbar_expect_tx(bars.a_full(), 2 * C::kTileBytes);
    load_tile<D>(sbase + BC::kOffA, &p.tm_q, bars.a_full(), q0, h, b);
    load_tile<D>(sbase + BC::kOffB, &bp.tm_do, bars.a_full(), q0, h, b);
    armed_a = 0;
    for (int j = band_next(band, -1); j < p.n_kv; j = band_next(band, j)) {
      if (tile_class<MASK>(q0, j, p) == 0) continue;
      const int s = static_cast<int>(it % BC::kStages);
      if (!warp_wait(bars.ring_empty(s), ((it / BC::kStages) & 1u) ^ 1u, ctl, j, kRoleLoader))
        goto ldrain;
      mbar_expect_tx(bars.ring_full(s), 2 * C::kTileBytes);
      load_tile<D>(sbase + BC::kOffRing + s * BC::kRingStride, &p.tm_k, bars.ring_full(s), j * kBN, h, b);
      load_tile<D>(sbase + BC::kOffRing + s * BC::kRingStride + C::kTileBytes, &p.tm_v,
                   bars.ring_full(s), j * kBN, h, b);
      armed[s] = static_cast<int>((it / BC::kStages) & 1u);
      ++it;
    }
  ldrain:
    if (armed_a >= 0) warp_wait(bars.a_full(), 0, ctl, -1, kRoleLoader, false);
    for (int s = 0; s < BC::kStages; ++s)
      if (armed[s] >= 0) warp_wait(bars.ring_full(s), armed[s], ctl, -1, kRoleLoader, false);
  } else if (warp == 1) {
    // per K/V tile: dQ += dS K of the previous tile, then S and dP of this one
    uint32_t it = 0, g_par = 0;
    int prev = -1;
    bool acc = false;
    if (!warp_wait(bars.a_full(), 0, ctl, -1, kRoleMma)) goto mdrain;
    tc_fence_after();
    for (int j = band_next(band, -1); j < p.n_kv; j = band_next(band, j)) {
      if (tile_class<MASK>(q0, j, p) == 0) continue;
      const int s = static_cast<int>(it % BC::kStages);
      if (!warp_wait(bars.ring_full(s), (it / BC::kStages) & 1u, ctl, j, kRoleMma)) goto mdrain;
      tc_fence_after();
      if (prev >= 0) {
        if (!warp_wait(bars.g_full(), g_par, ctl, j, kRoleMma)) goto mdrain;
        g_par ^= 1u;
        tc_fence_after();
        issue_tmn<D>(tmem + 256, tmem, sbase + BC::kOffRing + prev * BC::kRingStride, acc);
        acc = true;
        mma_commit(bars.ring_empty(prev));
      }
      const uint32_t kt = sbase + BC::kOffRing + s * BC::kRingStride;
      issue_nn<D>(tmem, sbase + BC::kOffA, kt);                               // S = Q K^T
      issue_nn<D>(tmem + 128, sbase + BC::kOffB, kt + C::kTileBytes);         // dP = dO V^T
      mma_commit(bars.s_full());
      prev = s;
      ++it;
    }
    if (prev >= 0) {
      if (!warp_wait(bars.g_full(), g_par, ctl, -1, kRoleMma)) goto mdrain;
      tc_fence_after();
      issue_tmn<D>(tmem + 256, tmem, sbase + BC::kOffRing + prev * BC::kRingStride, acc);
      mma_commit(bars.ring_empty(prev));
    }
    mma_commit(bars.acc_full());
  mdrain:
    mma_commit(bars.done());
    warp_wait(bars.done(), 0, ctl, -1, kRoleMma, false);
  } else if (warp >= 4) {
    // one thread per query row: P = exp(scale S - LSE), dS = P (dP - D)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int q = q0 + row;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool row_ok = q < p.Nq;
    const int64_t ri = static_cast<int64_t>(bh) * p.Nq + q;
    // a row that saw no key has LSE -inf: +inf here makes its P exactly 0
    const float lse_r = row_ok ? bp.lse[ri] : 0.f;
    const float lse2 = lse_r == -CUDART_INF_F ? CUDART_INF_F : lse_r * 1.44269504088896340736f;
    const float drow = row_ok ? bp.dd[ri] : 0.f;
    const NaQuery nq = na_query<MASK>(p, q);
    uint32_t s_par = 0;
    bool any = false;
    for (int j = band_next(band, -1); j < p.n_kv; j = band_next(band, j)) {
      const int cls = tile_class<MASK>(q0, j, p);
      if (cls == 0) continue;
      if (!warp_wait(bars.s_full(), s_par, ctl, j)) goto cdone;
      s_par ^= 1u;
      tc_fence_after();
      uint32_t bits[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      if (cls == 2) {
        uint32_t allk[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) allk[i] = 0u;
        mask_tile<MASK>(allk, p, j, q, nq);
        // mask_tile writes -inf bit patterns where a key is not allowed
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t m = 0u;
#pragma unroll
          for (int i = 0; i < 32; ++i) m |= (allk[32 * w + i] == 0u ? 1u : 0u) << i;
          bits[w] = m;
        }
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[64], pv[64];
        tmem_ld32(lane_base + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(lane_base + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_ld32(lane_base + 128 + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&pv[0]));
        tmem_ld32(lane_base + 128 + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&pv[32]));
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float ds2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 2 * i + u, col = 64 * half + e;
            const bool ok = (bits[col >> 5] >> (col & 31)) & 1u;
            const float pe = ok ? ex2(__uint_as_float(sv[e]) * p.c - lse2) : 0.f;
            ds2[u] = pe * (__uint_as_float(pv[e]) - drow);
          }
          pk[i] = pack_bf16(ds2[0], ds2[1]);
        }
        // dS over the first half of S: columns [32 * half, 32 * half + 32) were read above
        store_packed32(lane_base + 32 * half, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.g_full());
      any = true;
    }
    // dQ row: scale * accumulator (zero if the row attended no tile)
    {
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(bp.dq) + ri * D;
      if (any) {
        if (!warp_wait(bars.acc_full(), 0, ctl, -1)) goto cdone;
        tc_fence_after();
      }
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        if (any) tmem_ld32(lane_base + 256 + 32 * ch, ov);
        if (row_ok) {
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = any ? pack_bf16(__uint_as_float(ov[2 * i]) * bp.scale,
                                        __uint_as_float(ov[2 * i + 1]) * bp.scale)
                            : 0u;
          uint4* o4 = reinterpret_cast<uint4*>(dst + 32 * ch);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            o4[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
      }
    }
  cdone:;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ dK, dV

// Neighbourhood masks seen from a key: bit e set iff query q0 + e (< Nq) has
// key (ky, kx) in its window. Clamped windows are not symmetric at the grid's
// borders, so each query's window is placed and tested.
// Query coordinates c on an axis of length G whose window (w wide, dilation
// 1) holds key coordinate k: [lo, lo + len), circular when the axis wraps.
// Clamp: the window start clamp(c - w/2, 0, G - w) never decreases with c, so
// the c with start <= k <= start + w - 1 form one interval: [k - w/2, k + w/2]
// widened to the border where the start is pinned there. Wrap: [k - w/2, k + w/2].
template <bool WRAP>
__host__ __device__ __forceinline__ void na_axis_queries(int k, int G, int w, int& lo, int& len) {
  const int h = w >> 1;
  if (WRAP) {
    lo = k - h < 0 ? k - h + G : k - h;
    len = w;
    return;
  }
  const int c_max = k >= G - w ? G - 1 : k + h;
  const int c_min = k - w + 1 <= 0 ? 0 : k - h;
  lo = c_min;
  len = c_max - c_min + 1;
}

template <int MASK>
__host__ __device__ __forceinline__ void na_key_bits(const KernelParams& p, int q0, int kk,
                                            uint32_t (&bits)[4]) {
  bits[0] = bits[1] = bits[2] = bits[3] = 0u;
  const int n = min(kBM, p.Nq - q0);
  if constexpr (mask_is_na2(MASK) && !mask_na_dilated(MASK)) {
    // dilation 1: the queries that see the key form a row interval and a
    // column interval; set the columns line by line as the forward does
    constexpr bool WH = mask_na_wrap_rows(MASK), WW = mask_na_wrap_cols(MASK);
    const int W = p.grid_w;
    const int ky = kk / W, kx = kk - ky * W;
    int ylo, ylen, xlo, xlen;
    na_axis_queries<WH>(ky, p.grid_h, p.window_h, ylo, ylen);
    na_axis_queries<WW>(kx, W, p.window_w, xlo, xlen);
    int qy = q0 / W;
    int qx0 = q0 - qy * W;
    for (int i = 0; i < n; ++qy) {
      const int len = min(W - qx0, n - i);  // this line's columns [qx0, qx0 + len)
      int dy = qy - ylo;
      if (WH && dy < 0) dy += p.grid_h;
      if (dy >= 0 && dy < ylen) na_line_cols<WW, false>(bits, i - qx0, qx0, len, xlo, W, xlen, 1);
      i += len;
      qx0 = 0;
    }
  } else if constexpr (MASK == kMaskNa3) {
    const bool wd = (p.na_wrap & kNa3WrapDepth) != 0, wh = (p.na_wrap & kNa3WrapRows) != 0,
               ww = (p.na_wrap & kNa3WrapCols) != 0;
    if (p.dilation == 1) {
      // as for 2-D: an interval of query coordinates per axis, then lines
      const int W = p.grid_w, Gh = p.grid_h, plane = Gh * W;
      const int kt = kk / plane, ky = (kk - kt * plane) / W, kx = kk - kt * plane - ky * W;
      int tlo, tlen, ylo, ylen, xlo, xlen;
      if (wd) na_axis_queries<true>(kt, p.grid_d, p.window_d, tlo, tlen);
      else na_axis_queries<false>(kt, p.grid_d, p.window_d, tlo, tlen);
      if (wh) na_axis_queries<true>(ky, Gh, p.window_h, ylo, ylen);
      else na_axis_queries<false>(ky, Gh, p.window_h, ylo, ylen);
      if (ww) na_axis_queries<true>(kx, W, p.window_w, xlo, xlen);
      else na_axis_queries<false>(kx, W, p.window_w, xlo, xlen);
      const int r0 = q0 / W;
      int qt = r0 / Gh, qy = r0 - qt * Gh;
      int qx0 = q0 - r0 * W;
      for (int i = 0; i < n;) {
        const int len = min(W - qx0, n - i);
        int dt = qt - tlo, dy = qy - ylo;
        if (wd && dt < 0) dt += p.grid_d;
        if (wh && dy < 0) dy += Gh;
        if (dt >= 0 && dt < tlen && dy >= 0 && dy < ylen) {
          if (ww) na_line_cols<true, false>(bits, i - qx0, qx0, len, xlo, W, xlen, 1);
          else na_line_cols<false, false>(bits, i - qx0, qx0, len, xlo, W, xlen, 1);
        }
        i += len;
        qx0 = 0;
        if (++qy == Gh) {
          qy = 0;
          ++qt;
        }
      }
      return;
    }
    const int plane = p.grid_h * p.grid_w, dl = p.dilation;
    const int kt = kk / plane, ky = (kk - kt * plane) / p.grid_w, kx = kk - kt * plane - ky * p.grid_w;
    int qt = q0 / plane;
    int qy = (q0 - qt * plane) / p.grid_w;
    int qx = q0 - qt * plane - qy * p.grid_w;
    for (int e = 0; e < n; ++e) {
      if (na_in_rt(kt, na_first_rt(qt, p.grid_d, p.window_d, dl, wd), p.grid_d, p.window_d, dl, wd) &&
          na_in_rt(ky, na_first_rt(qy, p.grid_h, p.window_h, dl, wh), p.grid_h, p.window_h, dl, wh) &&
          na_in_rt(kx, na_first_rt(qx, p.grid_w, p.window_w, dl, ww), p.grid_w, p.window_w, dl, ww))
        bits[e >> 5] |= 1u << (e & 31);
      if (++qx == p.grid_w) {
        qx = 0;
        if (++qy == p.grid_h) {
          qy = 0;
          ++qt;
        }
      }
    }
  } else {
    constexpr bool WH = mask_na_wrap_rows(MASK), WW = mask_na_wrap_cols(MASK);
    constexpr bool DIL = mask_na_dilated(MASK);
    const int ky = kk / p.grid_w, kx = kk - ky * p.grid_w;
    int qy = q0 / p.grid_w;
    int qx = q0 - qy * p.grid_w;
    for (int e = 0; e < n; ++e) {
      const int fy = na_window_first<WH, DIL>(qy, p.grid_h, p.window_h, p.dilation);
      const int fx = na_window_first<WW, DIL>(qx, p.grid_w, p.window_w, p.dilation);
      if (na_in_window<WH, DIL>(ky, fy, p.grid_h, p.window_h, p.dilation) &&
          na_in_window<WW, DIL>(kx, fx, p.grid_w, p.window_w, p.dilation))
        bits[e >> 5] |= 1u << (e & 31);
      if (++qx == p.grid_w) {
        qx = 0;
        ++qy;
      }
    }
  }
}

// One CTA per (batch, head, 128-key K/V tile).
template <int D, int MASK>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dkv_kernel(const __grid_constant__ BwdParams bp) {
  using C = Cfg<D>;
  using BC = BwdCfg<D>;
  const KernelParams& p = bp.f;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BwdBars bars{sbase + BC::kOffBar, BC::kStages};
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + BC::kOffBar + 8 * bars.count());
  volatile uint32_t* abort_flag = tmem_slot + 1;
  const int bh = blockIdx.x / p.n_kv;
  const int j = blockIdx.x - bh * p.n_kv;
  const int k0 = j * kBN;
  const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
  const int n_qt = (p.Nq + kBM - 1) / kBM;
  const Band band = bwd_band<MASK>(k0, p.Nk, n_qt, p);  // Q tiles that may meet this K/V tile

  if (threadIdx.x == 0) {
    mbar_init(bars.a_full(), 1);
    mbar_init(bars.s_full(), 1);
    mbar_init(bars.g_full(), 4);
    mbar_init(bars.acc_full(), 1);
    mbar_init(bars.done(), 1);
    for (int s = 0; s < BC::kStages; ++s) {
      mbar_init(bars.ring_full(s), 2);  // the TMA bytes, and the loader's LSE / D vector stores
      mbar_init(bars.ring_empty(s), 1);
    }
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{abort_flag, p.status, p.timeout_ns};
  const uint32_t t_dv = 256, t_dk = 256 + D;

  if (warp == 0) {
    int armed_a = -1, armed[4] = {-1, -1, -1, -1};
    uint32_t it = 0;
    mbar_expect_tx(bars.a_full(), 2 * C::kTileBytes);
    load_tile<D>(sbase + BC::kOffA, &p.tm_k, bars.a_full(), k0, h, b);
    load_tile<D>(sbase + BC::kOffB, &p.tm_v, bars.a_full(), k0, h, b);
    armed_a = 0;
    for (int i = band_next(band, -1); i < n_qt; i = band_next(band, i)) {
      if (tile_class<MASK>(i * kBM, j, p) == 0) continue;
      const int s = static_cast<int>(it % BC::kStages);
      if (!warp_wait(bars.ring_empty(s), ((it / BC::kStages) & 1u) ^ 1u, ctl, i, kRoleLoader))
        goto ldrain;
      mbar_expect_tx(bars.ring_full(s), 2 * C::kTileBytes);
      load_tile<D>(sbase + BC::kOffRing + s * BC::kRingStride, &p.tm_q, bars.ring_full(s), i * kBM, h, b);
      load_tile<D>(sbase + BC::kOffRing + s * BC::kRingStride + C::kTileBytes, &bp.tm_do,
                   bars.ring_full(s), i * kBM, h, b);
      armed[s] = static_cast<int>((it / BC::kStages) & 1u);
      // per-query LSE (log2 units; +inf past Nq, so P = 0 there) and D
      float* vec = reinterpret_cast<float*>(smem + BC::kOffVec + s * BC::kVecBytes);
      for (int t = lane; t < kBM; t += 32) {
        const int q = i * kBM + t;
        const int64_t ri = static_cast<int64_t>(bh) * p.Nq + q;
        const float lr = q < p.Nq ? bp.lse[ri] : -CUDART_INF_F;  // no key or no row: P = 0
        vec[t] = lr == -CUDART_INF_F ? CUDART_INF_F : lr * 1.44269504088896340736f;
        vec[kBM + t] = q < p.Nq ? bp.dd[ri] : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.ring_full(s));
      ++it;
    }
  ldrain:
    if (armed_a >= 0) warp_wait(bars.a_full(), 0, ctl, -1, kRoleLoader, false);
    for (int s = 0; s < BC::kStages; ++s)
      if (armed[s] >= 0) warp_wait(bars.ring_full(s), armed[s], ctl, -1, kRoleLoader, false);
  } else if (warp == 1) {
    uint32_t it = 0, g_par = 0;
    int prev = -1;
    bool acc = false;
    if (!warp_wait(bars.a_full(), 0, ctl, -1, kRoleMma)) goto mdrain;
    tc_fence_after();
    for (int i = band_next(band, -1); i < n_qt; i = band_next(band, i)) {
      if (tile_class<MASK>(i * kBM, j, p) == 0) continue;
      const int s = static_cast<int>(it % BC::kStages);
      if (!warp_wait(bars.ring_full(s), (it / BC::kStages) & 1u, ctl, i, kRoleMma)) goto mdrain;
      tc_fence_after();
      if (prev >= 0) {
        if (!warp_wait(bars.g_full(), g_par, ctl, i, kRoleMma)) goto mdrain;
        g_par ^= 1u;
        tc_fence_after();
        const uint32_t pt = sbase + BC::kOffRing + prev * BC::kRingStride;
        issue_tmn<D>(tmem + t_dv, tmem, pt + C::kTileBytes, acc);   // dV += P^T dO
        issue_tmn<D>(tmem + t_dk, tmem + 128, pt, acc);             // dK += dS^T Q
        acc = true;
        mma_commit(bars.ring_empty(prev));
      }
      const uint32_t qt = sbase + BC::kOffRing + s * BC::kRingStride;
      issue_nn<D>(tmem, sbase + BC::kOffA, qt);                          // S^T = K Q^T
      issue_nn<D>(tmem + 128, sbase + BC::kOffB, qt + C::kTileBytes);    // dP^T = V dO^T
      mma_commit(bars.s_full());
      prev = s;
      ++it;
    }
    if (prev >= 0) {
      if (!warp_wait(bars.g_full(), g_par, ctl, -1, kRoleMma)) goto mdrain;
      tc_fence_after();
      const uint32_t pt = sbase + BC::kOffRing + prev * BC::kRingStride;
      issue_tmn<D>(tmem + t_dv, tmem, pt + C::kTileBytes, acc);
      issue_tmn<D>(tmem + t_dk, tmem + 128, pt, acc);
      mma_commit(bars.ring_empty(prev));
    }
    mma_commit(bars.acc_full());
  mdrain:
    mma_commit(bars.done());
    warp_wait(bars.done(), 0, ctl, -1, kRoleMma, false);
  } else if (warp >= 4) {
    // one thread per key row: P^T = exp(scale S^T - LSE), dS^T = P^T (dP^T - D)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int kk = k0 + row;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t s_par = 0, it = 0;
    bool any = false;
    for (int i = band_next(band, -1); i < n_qt; i = band_next(band, i)) {
      if (tile_class<MASK>(i * kBM, j, p) == 0) continue;
      const int s = static_cast<int>(it % BC::kStages);
      // the loader's vector stores are ordered by ring_full (already complete once S^T is)
      if (!warp_wait(bars.ring_full(s), (it / BC::kStages) & 1u, ctl, i)) goto cdone;
      if (!warp_wait(bars.s_full(), s_par, ctl, i)) goto cdone;
      s_par ^= 1u;
      ++it;
      tc_fence_after();
      const float* vec = reinterpret_cast<const float*>(smem + BC::kOffVec + s * BC::kVecBytes);
      const int q0 = i * kBM;
      // causal: query q sees key kk iff q >= kk; first allowed column of this tile
      const int first = mask_is_causal(MASK) ? kk - causal_shift<MASK>(p) - q0 : 0;
      uint32_t nab[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      if (mask_is_na(MASK)) na_key_bits<MASK>(p, q0, kk, nab);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t sv[64], pv[64];
        tmem_ld32(lane_base + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tmem_ld32(lane_base + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tmem_ld32(lane_base + 128 + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&pv[0]));
        tmem_ld32(lane_base + 128 + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&pv[32]));
        uint32_t pk[32], gk[32];
#pragma unroll
        for (int i2 = 0; i2 < 32; ++i2) {
          float pe2[2], ds2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int e = 2 * i2 + u, col = 64 * half + e;
            const bool ok = col >= first && ((nab[col >> 5] >> (col & 31)) & 1u);
            const float pe = ok ? ex2(__uint_as_float(sv[e]) * p.c - vec[col]) : 0.f;
            pe2[u] = pe;
            ds2[u] = pe * (__uint_as_float(pv[e]) - vec[kBM + col]);
          }
          pk[i2] = pack_bf16(pe2[0], pe2[1]);
          gk[i2] = pack_bf16(ds2[0], ds2[1]);
        }
        store_packed32(lane_base + 32 * half, pk);          // P^T over S^T
        store_packed32(lane_base + 128 + 32 * half, gk);    // dS^T over dP^T
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.g_full());
      any = true;
    }
    {
      if (any) {
        if (!warp_wait(bars.acc_full(), 0, ctl, -1)) goto cdone;
        tc_fence_after();
      }
      const bool row_ok = kk < p.Nk;
      const int64_t rk = static_cast<int64_t>(bh) * p.Nk + kk;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(which == 0 ? bp.dv : bp.dk) + rk * D;
        const float mul = which == 0 ? 1.f : bp.scale;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t ov[32];
          if (any) tmem_ld32(lane_base + (which == 0 ? t_dv : t_dk) + 32 * ch, ov);
          if (row_ok) {
            uint32_t packed[16];
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2)
              packed[i2] = any ? pack_bf16(__uint_as_float(ov[2 * i2]) * mul,
                                           __uint_as_float(ov[2 * i2 + 1]) * mul)
                               : 0u;
            uint4* o4 = reinterpret_cast<uint4*>(dst + 32 * ch);
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2)
              o4[i2] = make_uint4(packed[4 * i2], packed[4 * i2 + 1], packed[4 * i2 + 2],
                                  packed[4 * i2 + 3]);
          }
        }
      }
    }
  cdone:;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// The caller's stream and the second stream the dK/dV kernel runs on.
struct BwdStreams {
  cudaStream_t s, aux;
  cudaEvent_t fork, join;
};

template <int D, int MASK>
cudaError_t launch_bwd_mask(const BwdParams& bp, const BwdStreams& st) {
  const cudaStream_t s = st.s;
  const KernelParams& p = bp.f;
  const int smem = BwdCfg<D>::kSmemBytes > 116 * 1024 ? BwdCfg<D>::kSmemBytes : 116 * 1024;
  auto kq = attn_bwd_dq_kernel<D, MASK>;
  auto kkv = attn_bwd_dkv_kernel<D, MASK>;
  cudaError_t e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.Nq;
  bwd_rowdot_kernel<<<static_cast<unsigned>((rows + 255) / 256), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(bp.o), static_cast<const __nv_bfloat16*>(bp.dout), bp.dd,
      rows, D);
  const int n_qt = (p.Nq + kBM - 1) / kBM;
  // dQ and dK/dV need only D and the inputs: dK/dV on the second stream fills
  // the SMs that the last wave of dQ CTAs leaves idle, and the reverse.
  if ((e = cudaEventRecord(st.fork, s)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(st.aux, st.fork, 0)) != cudaSuccess) return e;
  kq<<<static_cast<unsigned>(p.B * p.H * n_qt), kBwdThreads, smem, s>>>(bp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  kkv<<<static_cast<unsigned>(p.B * p.H * p.n_kv), kBwdThreads, smem, st.aux>>>(bp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaEventRecord(st.join, st.aux)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(s, st.join, 0);
}

template <int D>
cudaError_t launch_bwd_dim(const BwdParams& bp, int mask, const BwdStreams& s) {
  switch (mask) {
    case kMaskNone: return launch_bwd_mask<D, kMaskNone>(bp, s);
    case kMaskCausal: return launch_bwd_mask<D, kMaskCausal>(bp, s);
    case kMaskCausalBR: return launch_bwd_mask<D, kMaskCausalBR>(bp, s);
    case kMaskNa + 0: return launch_bwd_mask<D, kMaskNa + 0>(bp, s);
    case kMaskNa + 1: return launch_bwd_mask<D, kMaskNa + 1>(bp, s);
    case kMaskNa + 2: return launch_bwd_mask<D, kMaskNa + 2>(bp, s);
    case kMaskNa + 3: return launch_bwd_mask<D, kMaskNa + 3>(bp, s);
    case kMaskNa + 4: return launch_bwd_mask<D, kMaskNa + 4>(bp, s);
    case kMaskNa + 5: return launch_bwd_mask<D, kMaskNa + 5>(bp, s);
    case kMaskNa + 6: return launch_bwd_mask<D, kMaskNa + 6>(bp, s);
    case kMaskNa + 7: return launch_bwd_mask<D, kMaskNa + 7>(bp, s);
    case kMaskNa3: return launch_bwd_mask<D, kMaskNa3>(bp, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dev
}  // namespace attn
