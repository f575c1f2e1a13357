// Selective-scan backward (ss_scan_bwd) for sm_103a: backpropagation through
// time through the diagonal SSM state, with the states rebuilt from the
// forward's chunk checkpoints instead of a stored [B, L, D, N] history.
//
// One CTA = 64 channels of one batch row at a time.  Chunks are visited from
// last to first; each chunk (a multiple of 16 steps) is walked twice:
//   pass A (tiles in order):   from the chunk's checkpoint, advance
//       h_t = a_t h_{t-1} + delta_t B_t x_t and park the state entering every
//       8-step window in shared memory;
//   pass B (tiles in reverse): per 8-step window, rebuild a_t and h_t from the
//       parked state into registers (one ex2 per cell), then run the adjoint
//       G_t = ds_t C_t + a_{t+1} G_{t+1} backwards through the window:
//         q_t = (a_t G_t) h_{t-1};  sum_n q_t A  and  sum_n G_t B_t  (-> ddelta, dx)
//         dA += q_t delta_t;  dB_t += G_t delta_t x_t;  dC_t += ds_t h_t.
//       The carry a_t G_t crosses windows, tiles and chunks in registers.
// Sums over n are warp reduce-scatters; dB_t and dC_t (sums over d) are
// reduced across lanes and warps, written as one partial per 64-channel tile
// to the workspace, and summed in fixed order by ss_bwd_reduce_kernel, as are
// the per-CTA partials of dA and dD.  No atomics: results are bitwise
// reproducible.
#include "scan_common.cuh"

namespace {

using namespace ssk;

__device__ unsigned g_bwd_err;

template <typename T, int N, int NSTG>
struct BwdSmem {
  alignas(128) T dlt[NSTG][kTT * kDT];
  alignas(128) T x[NSTG][kTT * kDT];
  alignas(128) T z[NSTG][kTT * kDT];
  alignas(128) T dy[NSTG][kTT * kDT];
  alignas(128) T Bm[NSTG][kTT * N];
  alignas(128) T Cm[NSTG][kTT * N];
  alignas(16) float dlt_f[kTT * kDT];
  alignas(16) float dx_f[kTT * kDT];  // delta * x
  alignas(16) float ds_f[kTT * kDT];  // dy * silu(z)
  alignas(16) float B_f[kTT * N];
  alignas(16) float C_f[kTT * N];
  alignas(16) float s_f[kTT * kDT];   // C_t . h_t
  alignas(16) float sA_f[kTT * kDT];  // sum_n q_t A log2(e)
  alignas(16) float sB_f[kTT * kDT];  // sum_n G_t B_t
  alignas(16) float dBC_w[Geo<N>::W][kTT][2 * N];
  alignas(16) float Dv_s[kDT];
  alignas(16) float dD_red[Geo<N>::NT][8];
  alignas(8) uint64_t full[NSTG];
};

template <typename T, int N, int NSTG>
constexpr size_t bwd_smem_bytes(int chunk) {
  return ((sizeof(BwdSmem<T, N, NSTG>) + 15) / 16) * 16 + (size_t)(chunk / kS) * 2 * Geo<N>::NT * sizeof(float4);
}

struct BwdParams {
  const float* A;
  const float* Dv;
  const float* ckpt;
  const float* dh_last;
  float* dx;
  float* ddelta;
  float* dz;
  float* dh0;
  float* ws_dBC;  // [ndt][B][L][2N]
  float* ws_dA;   // [gy][D][N]
  float* ws_dD;   // [gy][D]
  int B, L, D, chunk, nchunks;
};

template <int N, typename T, int NSTG>
__global__ void __launch_bounds__(Geo<N>::NT) scan_bwd_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tm_dlt,
                                                              const __grid_constant__ CUtensorMap tm_x,
                                                              const __grid_constant__ CUtensorMap tm_z,
                                                              const __grid_constant__ CUtensorMap tm_dy,
                                                              const __grid_constant__ CUtensorMap tm_B,
                                                              const __grid_constant__ CUtensorMap tm_C) {
  using G = Geo<N>;
  using AT = ActT<T>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  BwdSmem<T, N, NSTG>& S = *reinterpret_cast<BwdSmem<T, N, NSTG>*>(smem_raw);
  float4* bnd = reinterpret_cast<float4*>(smem_raw + ((sizeof(BwdSmem<T, N, NSTG>) + 15) / 16) * 16);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ng = lane % G::NG, cg = lane / G::NG;
  const int dl = warp * G::WC + cg * 2;
  const int d0 = blockIdx.x * kDT;
  const int dg = d0 + dl;
  const bool dvalid = dg < p.D;
  const int n0 = ng * 4;
  const int L = p.L;
  const int ntiles = (L + kTT - 1) / kTT;
  const int tpc = p.chunk / kTT;                        // tiles per full chunk
  const int ntl = ntiles - (p.nchunks - 1) * tpc;       // tiles in the last chunk
  const int per_b = 2 * ntiles;                         // items per batch row
  const int nb = (p.B - (int)blockIdx.y + (int)gridDim.y - 1) / (int)gridDim.y;
  const int nitems = nb * per_b;
  constexpr uint32_t kActBytes = kTT * kDT * AT::kBytes;
  constexpr uint32_t kBCBytes = kTT * N * AT::kBytes;

  float2 Ap[2][2];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (dvalid) {
        const float* a = p.A + (size_t)(dg + j) * N + n0 + 2 * q;
        Ap[j][q] = f2(a[0] * kLog2e, a[1] * kLog2e);
      } else {
        Ap[j][q] = f2(0.f, 0.f);
      }
    }
  for (int c = tid; c < kDT; c += G::NT) S.Dv_s[c] = (d0 + c < p.D) ? p.Dv[d0 + c] : 0.f;

  // item k -> (batch row, chunk, tile within chunk, pass)
  auto decode = [&](int k, int& b, int& kc, int& tl, bool& passB) {
    b = (int)blockIdx.y + (k / per_b) * (int)gridDim.y;
    const int q = k % per_b;
    if (q < 2 * ntl) {
      kc = p.nchunks - 1;
      passB = q >= ntl;
      tl = passB ? ntl - 1 - (q - ntl) : q;
    } else {
      const int q2 = q - 2 * ntl;
      kc = p.nchunks - 2 - q2 / (2 * tpc);
      const int r = q2 % (2 * tpc);
      passB = r >= tpc;
      tl = passB ? tpc - 1 - (r - tpc) : r;
    }
  };
  auto issue = [&](int k) {
    int b, kc, tl;
    bool passB;
    decode(k, b, kc, tl, passB);
    const int slot = k % NSTG;
    const int t0 = (kc * tpc + tl) * kTT;
    mbar_arrive_expect_tx(&S.full[slot], passB ? 4 * kActBytes + 2 * kBCBytes : 2 * kActBytes + kBCBytes);
    tma_load_3d(S.dlt[slot], &tm_dlt, &S.full[slot], d0, t0, b);
    tma_load_3d(S.x[slot], &tm_x, &S.full[slot], d0, t0, b);
    tma_load_2d(S.Bm[slot], &tm_B, &S.full[slot], t0 * N, b);
    if (passB) {
      tma_load_3d(S.z[slot], &tm_z, &S.full[slot], d0, t0, b);
      tma_load_3d(S.dy[slot], &tm_dy, &S.full[slot], d0, t0, b);
      tma_load_2d(S.Cm[slot], &tm_C, &S.full[slot], t0 * N, b);
    }
  };

  if (tid == 0) {
    prefetch_tmap(&tm_dlt); prefetch_tmap(&tm_x); prefetch_tmap(&tm_z);
    prefetch_tmap(&tm_dy); prefetch_tmap(&tm_B); prefetch_tmap(&tm_C);
    for (int s = 0; s < NSTG; ++s) mbar_init(&S.full[s], 1);
    fence_barrier_init();
    for (int k = 0; k < NSTG && k < nitems; ++k) issue(k);
  }
  __syncthreads();

  float2 h[2][2];              // pass-A running state
  float2 ga[2][2];             // a_{t+1} * G_{t+1}: the adjoint carried backwards
  float2 dA2[2][2];            // dA partial sums of the thread's cells
  float dDacc[8];              // dD partial sums of the epilogue channel group
#pragma unroll
  for (int j = 0; j < 2; ++j) dA2[j][0] = dA2[j][1] = f2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < 8; ++e) dDacc[e] = 0.f;

  for (int k = 0; k < nitems; ++k) {
    const int slot = k % NSTG;
    int b, kc, tl;
    bool passB;
    decode(k, b, kc, tl, passB);
    const int t0 = (kc * tpc + tl) * kTT;

    if (k % per_b == 0) {  // entering batch row b: the gradient arriving on h_{L-1}
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.dh_last != nullptr && dvalid)
          v = *reinterpret_cast<const float4*>(p.dh_last + ((size_t)b * p.D + dg + j) * N + n0);
        ga[j][0] = f2(v.x, v.y);
        ga[j][1] = f2(v.z, v.w);
      }
    }

    bool ok = true;
    if (tid == 0) ok = mbar_wait_bounded(&S.full[slot], (k / NSTG) & 1, kWaitLimitNs);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        atomicOr(&g_bwd_err, kErrTmaTimeout);
        for (int k2 = k; k2 < k + NSTG && k2 < nitems; ++k2)
          mbar_wait_bounded(&S.full[k2 % NSTG], (k2 / NSTG) & 1, 100000000ull);
      }
      return;
    }

    if (!passB) {
      // ------------------------------------------------ pass A: park window states
      if (tl == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (dvalid) v = *reinterpret_cast<const float4*>(p.ckpt + (((size_t)b * p.D + dg + j) * p.nchunks + kc) * N + n0);
          h[j][0] = f2(v.x, v.y);
          h[j][1] = f2(v.z, v.w);
        }
      }
      for (int gi = tid; gi < kTT * kDT / 8; gi += G::NT) {
        float dv[8], xv[8];
        AT::ld8(&S.dlt[slot][gi * 8], dv);
        AT::ld8(&S.x[slot][gi * 8], xv);
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[e] *= dv[e];
        float4* a = reinterpret_cast<float4*>(&S.dlt_f[gi * 8]);
        a[0] = make_float4(dv[0], dv[1], dv[2], dv[3]);
        a[1] = make_float4(dv[4], dv[5], dv[6], dv[7]);
        float4* c = reinterpret_cast<float4*>(&S.dx_f[gi * 8]);
        c[0] = make_float4(xv[0], xv[1], xv[2], xv[3]);
        c[1] = make_float4(xv[4], xv[5], xv[6], xv[7]);
      }
      for (int gi = tid; gi < kTT * N / 4; gi += G::NT) {
        float bv[4];
        AT::ld4(&S.Bm[slot][gi * 4], bv);
        reinterpret_cast<float4*>(S.B_f)[gi] = make_float4(bv[0], bv[1], bv[2], bv[3]);
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < kTT; ++r) {
        if (r % kS == 0) {
          const int sb = (tl * kTT + r) / kS;
          bnd[(sb * 2 + 0) * G::NT + tid] = make_float4(h[0][0].x, h[0][0].y, h[0][1].x, h[0][1].y);
          bnd[(sb * 2 + 1) * G::NT + tid] = make_float4(h[1][0].x, h[1][0].y, h[1][1].x, h[1][1].y);
        }
        const float2 dd = *reinterpret_cast<const float2*>(&S.dlt_f[r * kDT + dl]);
        const float2 xx = *reinterpret_cast<const float2*>(&S.dx_f[r * kDT + dl]);
        const float4 Bv = *reinterpret_cast<const float4*>(&S.B_f[r * N + n0]);
        const float2 B01 = f2(Bv.x, Bv.y), B23 = f2(Bv.z, Bv.w);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 dj = bc2(j ? dd.y : dd.x);
          const float2 xj = bc2(j ? xx.y : xx.x);
          h[j][0] = fma2(ex2_2(mul2(dj, Ap[j][0])), h[j][0], mul2(xj, B01));
          h[j][1] = fma2(ex2_2(mul2(dj, Ap[j][1])), h[j][1], mul2(xj, B23));
        }
      }
      __syncthreads();
      if (tid == 0 && k + NSTG < nitems) issue(k + NSTG);
      continue;
    }

    // -------------------------------------------------- pass B: adjoint sweep
    for (int gi = tid; gi < kTT * kDT / 8; gi += G::NT) {
      float dv[8], xv[8], zv[8], gv[8];
      AT::ld8(&S.dlt[slot][gi * 8], dv);
      AT::ld8(&S.x[slot][gi * 8], xv);
      AT::ld8(&S.z[slot][gi * 8], zv);
      AT::ld8(&S.dy[slot][gi * 8], gv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        xv[e] *= dv[e];
        gv[e] *= zv[e] * sigmoid(zv[e]);
      }
      float4* a = reinterpret_cast<float4*>(&S.dlt_f[gi * 8]);
      a[0] = make_float4(dv[0], dv[1], dv[2], dv[3]);
      a[1] = make_float4(dv[4], dv[5], dv[6], dv[7]);
      float4* c = reinterpret_cast<float4*>(&S.dx_f[gi * 8]);
      c[0] = make_float4(xv[0], xv[1], xv[2], xv[3]);
      c[1] = make_float4(xv[4], xv[5], xv[6], xv[7]);
      float4* s = reinterpret_cast<float4*>(&S.ds_f[gi * 8]);
      s[0] = make_float4(gv[0], gv[1], gv[2], gv[3]);
      s[1] = make_float4(gv[4], gv[5], gv[6], gv[7]);
    }
    for (int gi = tid; gi < kTT * N / 4; gi += G::NT) {
      float bv[4], cv[4];
      AT::ld4(&S.Bm[slot][gi * 4], bv);
      AT::ld4(&S.Cm[slot][gi * 4], cv);
      reinterpret_cast<float4*>(S.B_f)[gi] = make_float4(bv[0], bv[1], bv[2], bv[3]);
      reinterpret_cast<float4*>(S.C_f)[gi] = make_float4(cv[0], cv[1], cv[2], cv[3]);
    }
    __syncthreads();

    const int dsi = dsum_index(lane);
    const bool dsw = (lane & G::kDupMask) == 0;
    for (int sub = kTT / kS - 1; sub >= 0; --sub) {
      const int sb = tl * (kTT / kS) + sub;
      float2 hb[2][2];
      {
        const float4 v0 = bnd[(sb * 2 + 0) * G::NT + tid], v1 = bnd[(sb * 2 + 1) * G::NT + tid];
        hb[0][0] = f2(v0.x, v0.y); hb[0][1] = f2(v0.z, v0.w);
        hb[1][0] = f2(v1.x, v1.y); hb[1][1] = f2(v1.z, v1.w);
      }
      float2 av[kS][2][2], hv[kS][2][2];
      // rebuild the window: a_t and h_t in registers, C.h and dC on the way
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        const int r = sub * kS + i;
        const float2 dd = *reinterpret_cast<const float2*>(&S.dlt_f[r * kDT + dl]);
        const float2 xx = *reinterpret_cast<const float2*>(&S.dx_f[r * kDT + dl]);
        const float2 gg = *reinterpret_cast<const float2*>(&S.ds_f[r * kDT + dl]);
        const float4 Bv = *reinterpret_cast<const float4*>(&S.B_f[r * N + n0]);
        const float4 Cv = *reinterpret_cast<const float4*>(&S.C_f[r * N + n0]);
        const float2 B01 = f2(Bv.x, Bv.y), B23 = f2(Bv.z, Bv.w);
        const float2 C01 = f2(Cv.x, Cv.y), C23 = f2(Cv.z, Cv.w);
        float yj[2];
        float2 dc0, dc1;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 dj = bc2(j ? dd.y : dd.x);
          const float2 xj = bc2(j ? xx.y : xx.x);
          const float2 gj = bc2(j ? gg.y : gg.x);
          const float2 hp0 = i ? hv[i - 1][j][0] : hb[j][0];
          const float2 hp1 = i ? hv[i - 1][j][1] : hb[j][1];
          av[i][j][0] = ex2_2(mul2(dj, Ap[j][0]));
          av[i][j][1] = ex2_2(mul2(dj, Ap[j][1]));
          hv[i][j][0] = fma2(av[i][j][0], hp0, mul2(xj, B01));
          hv[i][j][1] = fma2(av[i][j][1], hp1, mul2(xj, B23));
          const float2 yy = fma2(C23, hv[i][j][1], mul2(C01, hv[i][j][0]));
          yj[j] = yy.x + yy.y;
          if (j == 0) {
            dc0 = mul2(gj, hv[i][0][0]);
            dc1 = mul2(gj, hv[i][0][1]);
          } else {
            dc0 = fma2(gj, hv[i][1][0], dc0);
            dc1 = fma2(gj, hv[i][1][1], dc1);
          }
        }
        if constexpr (G::NG == 4) {
          const bool up = ng & 2;
          float keep = up ? yj[1] : yj[0];
          keep += __shfl_xor_sync(0xffffffffu, up ? yj[0] : yj[1], 2);
          keep += __shfl_xor_sync(0xffffffffu, keep, 1);
          if ((ng & 1) == 0) S.s_f[r * kDT + dl + (ng >> 1)] = keep;
        } else if constexpr (G::NG == 2) {
          const bool up = ng & 1;
          float keep = up ? yj[1] : yj[0];
          keep += __shfl_xor_sync(0xffffffffu, up ? yj[0] : yj[1], 1);
          S.s_f[r * kDT + dl + ng] = keep;
        } else {
          *reinterpret_cast<float2*>(&S.s_f[r * kDT + dl]) = f2(yj[0], yj[1]);
        }
        const float dcs = dsum4<N>(dc0.x, dc0.y, dc1.x, dc1.y, lane);
        if (dsw) S.dBC_w[warp][r][N + n0 + dsi] = dcs;
      }
      // adjoint sweep backwards through the window
#pragma unroll
      for (int i = kS - 1; i >= 0; --i) {
        const int r = sub * kS + i;
        const float2 dd = *reinterpret_cast<const float2*>(&S.dlt_f[r * kDT + dl]);
        const float2 xx = *reinterpret_cast<const float2*>(&S.dx_f[r * kDT + dl]);
        const float2 gg = *reinterpret_cast<const float2*>(&S.ds_f[r * kDT + dl]);
        const float4 Bv = *reinterpret_cast<const float4*>(&S.B_f[r * N + n0]);
        const float4 Cv = *reinterpret_cast<const float4*>(&S.C_f[r * N + n0]);
        const float2 B01 = f2(Bv.x, Bv.y), B23 = f2(Bv.z, Bv.w);
        const float2 C01 = f2(Cv.x, Cv.y), C23 = f2(Cv.z, Cv.w);
        float sA[2], sB[2];
        float2 db0, db1;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 dj = bc2(j ? dd.y : dd.x);
          const float2 xj = bc2(j ? xx.y : xx.x);
          const float2 gj = bc2(j ? gg.y : gg.x);
          const float2 hp0 = i ? hv[i - 1][j][0] : hb[j][0];
          const float2 hp1 = i ? hv[i - 1][j][1] : hb[j][1];
          const float2 G0 = fma2(gj, C01, ga[j][0]);  // G_t
          const float2 G1 = fma2(gj, C23, ga[j][1]);
          ga[j][0] = mul2(av[i][j][0], G0);           // a_t G_t
          ga[j][1] = mul2(av[i][j][1], G1);
          const float2 q0 = mul2(ga[j][0], hp0);      // q_t = a_t G_t h_{t-1}
          const float2 q1 = mul2(ga[j][1], hp1);
          const float2 sa = fma2(q1, Ap[j][1], mul2(q0, Ap[j][0]));
          const float2 sbb = fma2(G1, B23, mul2(G0, B01));
          sA[j] = sa.x + sa.y;
          sB[j] = sbb.x + sbb.y;
          dA2[j][0] = fma2(q0, dj, dA2[j][0]);
          dA2[j][1] = fma2(q1, dj, dA2[j][1]);
          if (j == 0) {
            db0 = mul2(G0, xj);
            db1 = mul2(G1, xj);
          } else {
            db0 = fma2(G0, xj, db0);
            db1 = fma2(G1, xj, db1);
          }
        }
        // sums over n of the pair group: (sA0, sA1, sB0, sB1)
        if constexpr (G::NG == 4) {
          const bool up = ng & 2;
          float k0 = up ? sB[0] : sA[0], k1 = up ? sB[1] : sA[1];
          k0 += __shfl_xor_sync(0xffffffffu, up ? sA[0] : sB[0], 2);
          k1 += __shfl_xor_sync(0xffffffffu, up ? sA[1] : sB[1], 2);
          const bool up1 = ng & 1;
          float kk = up1 ? k1 : k0;
          kk += __shfl_xor_sync(0xffffffffu, up1 ? k0 : k1, 1);
          (up ? S.sB_f : S.sA_f)[r * kDT + dl + (ng & 1)] = kk;
        } else if constexpr (G::NG == 2) {
          const bool up = ng & 1;
          float k0 = up ? sB[0] : sA[0], k1 = up ? sB[1] : sA[1];
          k0 += __shfl_xor_sync(0xffffffffu, up ? sA[0] : sB[0], 1);
          k1 += __shfl_xor_sync(0xffffffffu, up ? sA[1] : sB[1], 1);
          *reinterpret_cast<float2*>(&(up ? S.sB_f : S.sA_f)[r * kDT + dl]) = f2(k0, k1);
        } else {
          *reinterpret_cast<float2*>(&S.sA_f[r * kDT + dl]) = f2(sA[0], sA[1]);
          *reinterpret_cast<float2*>(&S.sB_f[r * kDT + dl]) = f2(sB[0], sB[1]);
        }
        const float dbs = dsum4<N>(db0.x, db0.y, db1.x, db1.y, lane);
        if (dsw) S.dBC_w[warp][r][n0 + dsi] = dbs;
      }
    }
    __syncthreads();

    // dB_t, dC_t of this 64-channel tile: sum over warps in fixed order
    for (int e = tid; e < kTT * 2 * N; e += G::NT) {
      const int r = e / (2 * N), c = e % (2 * N);
      const int t = t0 + r;
      if (t < L) {
        float acc = S.dBC_w[0][r][c];
#pragma unroll
        for (int w = 1; w < G::W; ++w) acc += S.dBC_w[w][r][c];
        p.ws_dBC[(((size_t)blockIdx.x * p.B + b) * L + t) * (2 * N) + c] = acc;
      }
    }
    // per-(t, d) gradients
    for (int gi = tid; gi < kTT * kDT / 8; gi += G::NT) {
      const int r = gi / (kDT / 8), c8 = (gi % (kDT / 8)) * 8;
      const int t = t0 + r, d = d0 + c8;
      if (t < L && d < p.D) {
        float dv[8], xv[8], zv[8], gv[8], o0[8], o1[8], o2[8];
        AT::ld8(&S.dlt[slot][r * kDT + c8], dv);
        AT::ld8(&S.x[slot][r * kDT + c8], xv);
        AT::ld8(&S.z[slot][r * kDT + c8], zv);
        AT::ld8(&S.dy[slot][r * kDT + c8], gv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int o = r * kDT + c8 + e;
          const float Dd = S.Dv_s[c8 + e];
          const float sg = sigmoid(zv[e]);
          const float s = S.s_f[o] + Dd * xv[e];
          const float ds = S.ds_f[o];
          const float sB = S.sB_f[o];
          o0[e] = ds * Dd + dv[e] * sB;                      // dx
          o1[e] = S.sA_f[o] * kLn2 + xv[e] * sB;             // ddelta
          o2[e] = gv[e] * s * sg * (1.0f + zv[e] * (1.0f - sg));  // dz
          dDacc[e] += ds * xv[e];
        }
        const size_t off = ((size_t)b * L + t) * p.D + d;
        ActT<float>::st8(p.dx + off, o0);
        ActT<float>::st8(p.ddelta + off, o1);
        ActT<float>::st8(p.dz + off, o2);
      }
    }
    __syncthreads();
    if (tid == 0 && k + NSTG < nitems) issue(k + NSTG);

    if (kc == 0 && tl == 0 && p.dh0 != nullptr && dvalid) {  // last item of batch row b: ga = a_0 G_0
#pragma unroll
      for (int j = 0; j < 2; ++j)
        *reinterpret_cast<float4*>(p.dh0 + ((size_t)b * p.D + dg + j) * N + n0) =
            make_float4(ga[j][0].x, ga[j][0].y, ga[j][1].x, ga[j][1].y);
    }
  }

  // per-CTA partials of dA and dD (summed over this CTA's batch rows)
  if (dvalid) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      *reinterpret_cast<float4*>(p.ws_dA + ((size_t)blockIdx.y * p.D + dg + j) * N + n0) =
          make_float4(dA2[j][0].x, dA2[j][0].y, dA2[j][1].x, dA2[j][1].y);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) S.dD_red[tid][e] = dDacc[e];
  __syncthreads();
  for (int c = tid; c < kDT; c += G::NT) {
    if (d0 + c < p.D) {
      const int grp = c / 8, e = c % 8;
      float acc = 0.f;
      for (int m = grp; m < G::NT; m += kDT / 8) acc += S.dD_red[m][e];
      p.ws_dD[(size_t)blockIdx.y * p.D + d0 + c] = acc;
    }
  }
}

// dB, dC = sum over channel tiles (overwrite); dA, dD += sum over CTA rows.
template <int N>
__global__ void ss_bwd_reduce_kernel(const float* __restrict__ ws_dBC, const float* __restrict__ ws_dA,
                                     const float* __restrict__ ws_dD, float* dB, float* dC, float* dA, float* dD, int B,
                                     int L, int D, int ndt, int gy) {
  const long long nBC = (long long)B * L * 2 * N;
  const long long nA = (long long)D * N;
  const long long total = nBC + nA + D;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    if (i < nBC) {
      float acc = 0.f;
      for (int t = 0; t < ndt; ++t) acc += ws_dBC[(size_t)t * nBC + i];
      const long long row = i / (2 * N);
      const int c = (int)(i % (2 * N));
      if (c < N) dB[row * N + c] = acc;
      else dC[row * N + (c - N)] = acc;
    } else if (i < nBC + nA) {
      const long long j = i - nBC;
      float acc = 0.f;
      for (int g = 0; g < gy; ++g) acc += ws_dA[(size_t)g * nA + j];
      dA[j] += acc;
    } else {
      const long long j = i - nBC - nA;
      float acc = 0.f;
      for (int g = 0; g < gy; ++g) acc += ws_dD[(size_t)g * D + j];
      dD[j] += acc;
    }
  }
}

struct BwdPlan {
  int ndt, gy;
  size_t off_dA, off_dD, total;
};

inline BwdPlan make_plan(int B, int L, int D, int N) {
  BwdPlan pl;
  pl.ndt = (D + kDT - 1) / kDT;
  const int cap = 1024 / pl.ndt > 0 ? 1024 / pl.ndt : 1;
  pl.gy = B < cap ? B : cap;
  const size_t bc = (size_t)pl.ndt * B * L * 2 * N * sizeof(float);
  pl.off_dA = (bc + 255) & ~(size_t)255;
  const size_t a = (size_t)pl.gy * D * N * sizeof(float);
  pl.off_dD = (pl.off_dA + a + 255) & ~(size_t)255;
  pl.total = pl.off_dD + (size_t)pl.gy * D * sizeof(float);
  return pl;
}

// pipeline depth: fp32 tiles are twice the size of bf16 ones
template <typename T>
struct Stages {
  static constexpr int value = sizeof(T) == 4 ? 2 : 3;
};

template <int N, typename T>
size_t bwd_smem(int chunk) {
  return bwd_smem_bytes<T, N, Stages<T>::value>(chunk);
}

template <int N, typename T>
int launch_bwd(BwdParams p, const void* x, const void* delta, const void* Bm, const void* Cm, const void* z, const void* dy,
               float* dA, float* dB, float* dC, float* dD, void* ws, cudaStream_t stream) {
  constexpr int e = ActT<T>::kBytes;
  constexpr int NSTG = Stages<T>::value;
  const BwdPlan pl = make_plan(p.B, p.L, p.D, N);
  p.ws_dBC = static_cast<float*>(ws);
  p.ws_dA = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.off_dA);
  p.ws_dD = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.off_dD);
  CUtensorMap tm[6];
  const uint64_t adims[3] = {(uint64_t)p.D, (uint64_t)p.L, (uint64_t)p.B};
  const uint64_t astr[2] = {(uint64_t)p.D * e, (uint64_t)p.L * p.D * e};
  const uint32_t abox[3] = {kDT, kTT, 1};
  const uint64_t bdims[2] = {(uint64_t)p.L * N, (uint64_t)p.B};
  const uint64_t bstr[1] = {(uint64_t)p.L * N * e};
  const uint32_t bbox[2] = {kTT * N, 1};
  if (!ssh::encode_tiled(&tm[0], ActT<T>::kTma, 3, delta, adims, astr, abox) ||
      !ssh::encode_tiled(&tm[1], ActT<T>::kTma, 3, x, adims, astr, abox) ||
      !ssh::encode_tiled(&tm[2], ActT<T>::kTma, 3, z, adims, astr, abox) ||
      !ssh::encode_tiled(&tm[3], ActT<T>::kTma, 3, dy, adims, astr, abox) ||
      !ssh::encode_tiled(&tm[4], ActT<T>::kTma, 2, Bm, bdims, bstr, bbox) ||
      !ssh::encode_tiled(&tm[5], ActT<T>::kTma, 2, Cm, bdims, bstr, bbox))
    return SS_ERR_CUDA;
  const size_t smem = bwd_smem<N, T>(p.chunk);
  auto kern = scan_bwd_kernel<N, T, NSTG>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return SS_ERR_CUDA;
  kern<<<dim3(pl.ndt, pl.gy), Geo<N>::NT, smem, stream>>>(p, tm[0], tm[1], tm[2], tm[3], tm[4], tm[5]);
  if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
  const long long total = (long long)p.B * p.L * 2 * N + (long long)p.D * N + p.D;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  ss_bwd_reduce_kernel<N><<<(int)blocks, 256, 0, stream>>>(p.ws_dBC, p.ws_dA, p.ws_dD, dB, dC, dA, dD, p.B, p.L, p.D,
                                                           pl.ndt, pl.gy);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

constexpr size_t kMaxSmem = 227 * 1024;

bool bwd_chunk_fits(int N, int dtype, int chunk) {
  size_t s;
  if (dtype == SS_F32) s = N == 4 ? bwd_smem<4, float>(chunk) : N == 8 ? bwd_smem<8, float>(chunk) : bwd_smem<16, float>(chunk);
  else s = N == 4 ? bwd_smem<4, __nv_bfloat16>(chunk) : N == 8 ? bwd_smem<8, __nv_bfloat16>(chunk) : bwd_smem<16, __nv_bfloat16>(chunk);
  return s <= kMaxSmem;
}

int validate_bwd(int B, int L, int D, int N, int chunk, int dtype) {
  if (B <= 0 || L <= 0 || D <= 0 || N <= 0 || chunk <= 0) return SS_ERR_DIM;
  if (N != 4 && N != 8 && N != 16) return SS_ERR_UNSUPPORTED;
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (chunk % kTT != 0 || !bwd_chunk_fits(N, dtype, chunk)) return SS_ERR_UNSUPPORTED;
  if (D % 8 != 0) return SS_ERR_ALIGN;
  if (((long long)L * N * (dtype == SS_F32 ? 4 : 2)) % 16 != 0) return SS_ERR_ALIGN;
  if ((long long)L * N >= (1ll << 31) || (long long)L * D >= (1ll << 40)) return SS_ERR_DIM;
  return SS_OK;
}

}  // namespace

namespace ssh {
int read_clear_bwd_err(cudaStream_t s, unsigned* out) {
  unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(out, g_bwd_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SS_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_bwd_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s) != cudaSuccess) return SS_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
}  // namespace ssh

extern "C" size_t ss_scan_bwd_workspace_size(int B, int L, int D, int N, int chunk, int dtype) {
  if (validate_bwd(B, L, D, N, chunk, dtype) != SS_OK) return 0;
  return make_plan(B, L, D, N).total;
}

extern "C" int ss_scan_bwd(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm, const float* Dv,
                           const void* z, const float* ckpt, const void* dy, const float* dh_last, float* dx, float* ddelta,
                           float* dz, float* dA, float* dB, float* dC, float* dD, float* dh0, int B, int L, int D, int N,
                           int chunk, int dtype, void* workspace, size_t ws_bytes, void* stream) {
  if (!x || !delta || !A || !Bm || !Cm || !Dv || !z || !ckpt || !dy || !dx || !ddelta || !dz || !dA || !dB || !dC || !dD)
    return SS_ERR_NULL;
  const int v = validate_bwd(B, L, D, N, chunk, dtype);
  if (v != SS_OK) return v;
  const void* ptrs[] = {x, delta, A, Bm, Cm, Dv, z, ckpt, dy, dx, ddelta, dz, dA, dB, dC, dD};
  for (const void* q : ptrs)
    if (!ssh::aligned16(q)) return SS_ERR_ALIGN;
  if ((dh_last && !ssh::aligned16(dh_last)) || (dh0 && !ssh::aligned16(dh0))) return SS_ERR_ALIGN;
  const BwdPlan pl = make_plan(B, L, D, N);
  if (workspace == nullptr || ws_bytes < pl.total) return SS_ERR_WORKSPACE;
  if (!ssh::aligned16(workspace)) return SS_ERR_ALIGN;
  BwdParams p{A, Dv, ckpt, dh_last, dx, ddelta, dz, dh0, nullptr, nullptr, nullptr, B, L, D, chunk, ss_scan_num_chunks(L, chunk)};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SS_F32) {
    if (N == 4) return launch_bwd<4, float>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
    if (N == 8) return launch_bwd<8, float>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
    return launch_bwd<16, float>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
  }
  if (N == 4) return launch_bwd<4, __nv_bfloat16>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
  if (N == 8) return launch_bwd<8, __nv_bfloat16>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
  return launch_bwd<16, __nv_bfloat16>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
}
