// Selective-scan forward (ss_scan_fwd) for sm_103a.
//
//   h_t = exp(delta_t * A) * h_{t-1} + delta_t * B_t * x_t,   y_t = (C_t . h_t + D x_t) * silu(z_t)
//
// Main kernel: one CTA = one warp = CG channels of one batch row (CG = 32 /
// (N/4)).  Lane (ng, c) owns channel c and states 4ng .. 4ng+3: four (d, n)
// recurrences in registers, f32x2-packed, with one ex2 per (t, d, n) (A
// pre-scaled by log2 e).  The sequence is walked once, in order, in 16-step
// tiles that TMA stages into a ring (2 deep for bf16, 3 for fp32).  The
// recurrence reads delta and x straight from the staging slot; B_t and C_t,
// shared by every lane of a state quad, are widened to fp32 once per tile so
// that each step loads them with one 128-bit broadcast read.  C_t . h_t is
// summed over the N/4 lanes of a channel by a shuffle reduce-scatter over four
// steps (two when N = 8), after which every lane holds the complete sum of one
// (t, d) and forms y = (s + D x) * silu(z) itself.  A warp needs no block barrier: copies are
// observed on mbarriers and slot reuse is ordered by warp syncs, so the ~13
// warps an SM holds on a Mamba-sized layer never wait on one another.
// The state entering step c*chunk is stored as checkpoint c ([B, chunks, D, N])
// for the backward.
//
// Sequence segments (few batch rows, long sequences): a summary kernel gives
// each segment's zero-start end state and its sum of delta; a combine kernel
// composes the segments' affine maps h -> exp2(A' sum delta) h + end state
// with a warp-shuffle associative scan and writes the state entering every
// segment; the main kernel then runs each segment from its carry.
#include "scan_common.cuh"

namespace {

using namespace ssk;

__device__ unsigned g_fwd_err;

// TMA pipeline depth (tiles in flight per one-warp CTA).  Fewer slots leave
// room for more resident CTAs, which the segment and grid choices turn into
// parallelism: two for bf16, three for fp32 (against four: long-context
// forward 361 -> 332 us, short many-batch 67 -> 60 / 64 us, mamba130m
// 212 -> 205 us with three, the 1.4B layer unchanged).
template <typename T>
constexpr int fwd_stages() {
  return sizeof(T) == 2 ? 2 : 3;
}

struct FwdParams {
  const float* A;
  const float* Dv;
  const float* h0;
  void* y;
  float* ckpt;
  float* h_last;
  int B, L, D, chunk, nchunks;
  int P, Ls;     // sequence segments (P = 1: one CTA row walks whole batch rows)
  float* hsum;   // [B][P][D][N] state at the end of each segment from a zero start
  float* dsum;   // [B][P][D]    sum of delta over each segment
  float* hin;    // [B][P][D][N] state entering each segment (combine kernel output)
  int sum_stride;  // summary pass: rows of hsum / dsum per batch row (P inside ss_scan_fwd, 1 for one whole sequence)
  const float* dt_bias;  // fused discretisation: delta = f(raw + dt_bias), f = softplus if dsp
  int dsp;
  int fuse;              // dt_bias != NULL or dsp
};

// Main-kernel geometry: one warp per CTA, one channel x 4 states per lane, CG = 32 / (N/4) channels.
template <int N>
struct GeoW {
  static constexpr int NG = N / 4;
  static constexpr int CG = 32 / NG;
  static constexpr int DT = CG;
};

template <typename T, int N>
struct FwdSmem {
  static constexpr int DT = GeoW<N>::DT;
  static constexpr int kNST = fwd_stages<T>();
  alignas(128) T dlt[kNST][kTT * DT];
  alignas(128) T x[kNST][kTT * DT];
  alignas(128) T z[kNST][kTT * DT];
  alignas(128) T Bm[kNST][kTT * N];
  alignas(128) T Cm[kNST][kTT * N];
  alignas(16) float dlt_f[kTT * DT];  // fused discretisation only: the tile's transformed delta
  alignas(16) float B_f[kTT * N];     // the tile's B_t, C_t in fp32
  alignas(16) float C_f[kTT * N];
  alignas(16) float bias_s[DT];
  alignas(8) uint64_t full[kNST];
};

// SUM = true: the segment-summary pass.  CTA row y = (batch row, segment) for
// segments 0 .. P-2, which are whole tiles; only delta, x and B_t are read and
// the kernel writes the segment's end state from a zero start and its sum of delta.
template <int N, typename T, bool FUSE, bool SUM>
__global__ void __launch_bounds__(32) scan_fwd_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_dlt,
                                                       const __grid_constant__ CUtensorMap tm_x,
                                                       const __grid_constant__ CUtensorMap tm_z,
                                                       const __grid_constant__ CUtensorMap tm_B,
                                                       const __grid_constant__ CUtensorMap tm_C) {
  using G = GeoW<N>;
  using AT = ActT<T>;
  constexpr int NG = G::NG, CG = G::CG, DT = G::DT;
  constexpr int kNST = FwdSmem<T, N>::kNST;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  FwdSmem<T, N>& S = *reinterpret_cast<FwdSmem<T, N>*>(smem_raw);

  const int lane = threadIdx.x;
  const int ng = lane / CG, c = lane % CG;
  const int n0 = ng * 4;
  const int d0 = blockIdx.x * DT;
  const int dg = d0 + c;
  const bool dvalid = dg < p.D;
  const int L = p.L;
  const bool segs = SUM || p.P > 1;
  const int sgm = SUM ? (int)blockIdx.y % (p.P - 1) : segs ? (int)blockIdx.y % p.P : 0;
  const int tb = sgm * p.Ls;
  const int te = segs ? min(L, tb + p.Ls) : L;
  const int ntiles = (te - tb + kTT - 1) / kTT;
  const int nb = segs ? 1 : (p.B - (int)blockIdx.y + (int)gridDim.y - 1) / (int)gridDim.y;
  const int nitems = nb * ntiles;
  const int b_first = SUM ? (int)blockIdx.y / (p.P - 1) : segs ? (int)blockIdx.y / p.P : (int)blockIdx.y;
  struct Cursor {
    int b, ti;
  };
  auto advance = [&](Cursor& cu) {
    if (++cu.ti == ntiles) {
      cu.ti = 0;
      cu.b += (int)gridDim.y;
    }
  };
  Cursor icur{b_first, 0};
  constexpr uint32_t kStageBytes = (SUM ? 2 : 3) * kTT * DT * AT::kBytes + (SUM ? 1 : 2) * kTT * N * AT::kBytes;

  float2 Ap[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float* a = p.A + (size_t)(dvalid ? dg : 0) * N + n0 + 2 * q;
    Ap[q] = dvalid ? f2(a[0] * kLog2e, a[1] * kLog2e) : f2(0.f, 0.f);
  }
  const float Dc = dvalid ? p.Dv[dg] : 0.f;
  if constexpr (FUSE)
    for (int i = lane; i < DT; i += 32) S.bias_s[i] = (p.dt_bias != nullptr && d0 + i < p.D) ? p.dt_bias[d0 + i] : 0.f;

  auto issue = [&](int k) {
    fence_proxy_async_smem();
    const int slot = k % kNST;
    const int bb = icur.b;
    const int t0 = tb + icur.ti * kTT;
    advance(icur);
    mbar_arrive_expect_tx(&S.full[slot], kStageBytes);
    tma_load_3d(S.dlt[slot], &tm_dlt, &S.full[slot], d0, t0, bb);
    tma_load_3d(S.x[slot], &tm_x, &S.full[slot], d0, t0, bb);
    tma_load_2d(S.Bm[slot], &tm_B, &S.full[slot], t0 * N, bb);
    if constexpr (!SUM) {
      tma_load_3d(S.z[slot], &tm_z, &S.full[slot], d0, t0, bb);
      tma_load_2d(S.Cm[slot], &tm_C, &S.full[slot], t0 * N, bb);
    }
  };
  if (lane == 0) {
    prefetch_tmap(&tm_dlt); prefetch_tmap(&tm_x); prefetch_tmap(&tm_z); prefetch_tmap(&tm_B); prefetch_tmap(&tm_C);
    for (int s = 0; s < kNST; ++s) mbar_init(&S.full[s], 1);
    fence_barrier_init();
    for (int k = 0; k < kNST && k < nitems; ++k) issue(k);
  }
  __syncwarp();

  // y at step r of the tile for this lane's channel, from its sum over n
  auto finish1 = [&](int slot, int b, int t0, int r, float sv) {
    const float xv = AT::ld(&S.x[slot][r * DT + c]);
    const float zv = AT::ld(&S.z[slot][r * DT + c]);
    const float o = fmaf(Dc, xv, sv) * zv * sigmoid(zv);
    if (t0 + r < L && dvalid) AT::st1(reinterpret_cast<T*>(p.y) + ((size_t)b * L + t0 + r) * p.D + dg, o);
  };

  float2 h0, h1;
  float dsum = 0.f;  // SUM: the segment's sum of delta
  Cursor cur{b_first, 0};
  int tck = 0;
  for (int k = 0; k < nitems; ++k, advance(cur)) {
    const int slot = k % kNST;
    const int b = cur.b;
    const int ti = cur.ti;
    const int t0 = tb + ti * kTT;
    if (ti == 0) {
      tck = tb % p.chunk;
      const float* src = SUM ? nullptr
                             : segs ? p.hin + ((size_t)b * p.P + sgm) * p.D * N : (p.h0 ? p.h0 + (size_t)b * p.D * N : nullptr);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (src != nullptr && dvalid) v = *reinterpret_cast<const float4*>(src + (size_t)dg * N + n0);
      h0 = f2(v.x, v.y);
      h1 = f2(v.z, v.w);
    }
    const bool ok = mbar_wait_bounded(&S.full[slot], (k / kNST) & 1, kWaitLimitNs);
    if (__any_sync(0xffffffffu, !ok)) {
      if (lane == 0) {
        atomicOr(&g_fwd_err, kErrTmaTimeout);
        for (int k2 = k; k2 < k + kNST && k2 < nitems; ++k2)
          mbar_wait_bounded(&S.full[k2 % kNST], (k2 / kNST) & 1, 100000000ull);
      }
      return;
    }
    if constexpr (FUSE) {
      for (int gi = lane; gi < kTT * DT / 4; gi += 32) {
        float dv[4];
        AT::ld4(&S.dlt[slot][gi * 4], dv);
        const int c4 = (gi % (DT / 4)) * 4;
        delta_transform4(dv, S.bias_s, c4, t0 + gi / (DT / 4) < L, p.D - d0 - c4, p.dsp);
        *reinterpret_cast<float4*>(&S.dlt_f[gi * 4]) = make_float4(dv[0], dv[1], dv[2], dv[3]);
      }
    }
    for (int gi = lane; gi < kTT * N / 4; gi += 32) {
      float bv[4];
      AT::ld4(&S.Bm[slot][gi * 4], bv);
      reinterpret_cast<float4*>(S.B_f)[gi] = make_float4(bv[0], bv[1], bv[2], bv[3]);
      if constexpr (!SUM) {
        float cv[4];
        AT::ld4(&S.Cm[slot][gi * 4], cv);
        reinterpret_cast<float4*>(S.C_f)[gi] = make_float4(cv[0], cv[1], cv[2], cv[3]);
      }
    }
    __syncwarp();
#pragma unroll
    for (int rq = 0; rq < kTT; rq += 4) {
      float ys[4];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int r = rq + s;
        if (!SUM && (r == 0 || r == kS)) {
          const int tc = t0 + r;
          if (dvalid && tc < L && (p.chunk == kS || (r == 0 && tck == 0))) {
            const int ci = p.chunk == kS ? tc / kS : tc / p.chunk;
            *reinterpret_cast<float4*>(p.ckpt + (((size_t)b * p.nchunks + ci) * p.D + dg) * N + n0) =
                make_float4(h0.x, h0.y, h1.x, h1.y);
          }
        }
        float dv;
        if constexpr (FUSE) dv = S.dlt_f[r * DT + c];
        else dv = AT::ld(&S.dlt[slot][r * DT + c]);
        const float uv = dv * AT::ld(&S.x[slot][r * DT + c]);
        float2 B01, B23;
        ActT<float>::ld4x2(&S.B_f[r * N + n0], B01, B23);
        const float2 d2 = bc2(dv), u2 = bc2(uv);
        h0 = fma2(ex2_2(mul2(d2, Ap[0])), h0, mul2(u2, B01));
        h1 = fma2(ex2_2(mul2(d2, Ap[1])), h1, mul2(u2, B23));
        if constexpr (SUM) {
          dsum += dv;
          continue;
        }
        float2 C01, C23;
        ActT<float>::ld4x2(&S.C_f[r * N + n0], C01, C23);
        const float2 yy = fma2(C23, h1, mul2(C01, h0));
        ys[s] = yy.x + yy.y;
        if constexpr (NG == 1) {
          finish1(slot, b, t0, r, ys[s]);
        } else if constexpr (NG == 2) {
          if (s & 1) finish1(slot, b, t0, r - 1 + (ng & 1), rs_pair(ys[s - 1], ys[s], ng & 1, CG));
        }
      }
      if constexpr (NG == 4 && !SUM) {  // the four steps: keep steps {2 b1, 2 b1 + 1}, then step ng
        const bool b1 = (ng >> 1) & 1, b0 = ng & 1;
        const float k0 = rs_pair(ys[0], ys[2], b1, 2 * CG);
        const float k1 = rs_pair(ys[1], ys[3], b1, 2 * CG);
        finish1(slot, b, t0, rq + ng, rs_pair(k0, k1, b0, CG));
      }
    }
    tck += kTT;
    if (tck >= p.chunk) tck -= p.chunk;
    __syncwarp();
    if (lane == 0 && k + kNST < nitems) issue(k + kNST);
    if (!SUM && ti == ntiles - 1 && te == L && p.h_last != nullptr && dvalid)
      *reinterpret_cast<float4*>(p.h_last + ((size_t)b * p.D + dg) * N + n0) = make_float4(h0.x, h0.y, h1.x, h1.y);
  }
  if (SUM && dvalid) {
    const size_t row = ((size_t)b_first * p.sum_stride + sgm) * p.D + dg;
    *reinterpret_cast<float4*>(p.hsum + row * N + n0) = make_float4(h0.x, h0.y, h1.x, h1.y);
    if (ng == 0) p.dsum[row] = dsum;
  }
}

// Segments only when the (batch row, channel tile) warps would leave the GPU
// with fewer than four per SM.
template <int N>
int fwd_pmax(int B, int L, int D) {
  constexpr int DT = GeoW<N>::DT;
  const long long warps = (long long)((D + DT - 1) / DT) * B;
  return warps >= 608 ? 1 : seg_pmax(warps, L, kTT, 32 * 152);  // one-warp CTAs: aim at 32 per SM
}

struct FwdWs {
  size_t off_dsum, off_hin, total;
};

inline FwdWs fwd_ws_layout(int B, int D, int N, int pm) {
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  const size_t st = (size_t)B * pm * D * N * sizeof(float);
  FwdWs w;
  w.off_dsum = up(st);
  w.off_hin = up(w.off_dsum + (size_t)B * pm * D * sizeof(float));
  w.total = w.off_hin + st;
  return w;
}

size_t fwd_ws_bytes(int B, int L, int D, int N) {
  const int pm = N == 4 ? fwd_pmax<4>(B, L, D) : N == 8 ? fwd_pmax<8>(B, L, D) : fwd_pmax<16>(B, L, D);
  if (pm <= 1) return 0;
  return fwd_ws_layout(B, D, N, pm).total;
}

template <int N, typename T, bool FUSE>
int launch_fwd(FwdParams p, const void* x, const void* delta, const void* Bm, const void* Cm, const void* z, void* ws,
               cudaStream_t stream) {
  constexpr int e = ActT<T>::kBytes;
  constexpr int DT = GeoW<N>::DT;
  CUtensorMap tm[5];
  const uint64_t adims[3] = {(uint64_t)p.D, (uint64_t)p.L, (uint64_t)p.B};
  const uint64_t astr[2] = {(uint64_t)p.D * e, (uint64_t)p.L * p.D * e};
  const uint32_t abox[3] = {DT, kTT, 1};
  const uint64_t bdims[2] = {(uint64_t)p.L * N, (uint64_t)p.B};
  const uint64_t bstr[1] = {(uint64_t)p.L * N * e};
  const uint32_t bbox[2] = {kTT * N, 1};
  if (!ssh::encode_tiled(&tm[0], ActT<T>::kTma, 3, delta, adims, astr, abox) ||
      !ssh::encode_tiled(&tm[1], ActT<T>::kTma, 3, x, adims, astr, abox) ||
      !ssh::encode_tiled(&tm[2], ActT<T>::kTma, 3, z, adims, astr, abox) ||
      !ssh::encode_tiled(&tm[3], ActT<T>::kTma, 2, Bm, bdims, bstr, bbox) ||
      !ssh::encode_tiled(&tm[4], ActT<T>::kTma, 2, Cm, bdims, bstr, bbox))
    return SS_ERR_CUDA;
  const int ndt = (p.D + DT - 1) / DT;
  const size_t smem = sizeof(FwdSmem<T, N>);
  auto kern = scan_fwd_kernel<N, T, FUSE, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return SS_ERR_CUDA;
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  // segments: only when (batch row, channel tile) warps leave SMs idle
  p.P = 1;
  p.Ls = p.L;
  const int pmax = fwd_pmax<N>(p.B, p.L, p.D);
  if (pmax > 1) {
    const int per_sm = resident_ctas(kern, 32, smem);
    if (per_sm < 1) return SS_ERR_CUDA;
    const long long resident = (long long)per_sm * device_sm_count();
    int want = (int)(resident / ((long long)ndt * p.B));
    if (want > pmax) want = pmax;
    const SegPlan sp = seg_plan(want, p.L, kTT);
    p.P = sp.P;
    p.Ls = sp.Ls;
    p.sum_stride = sp.P;
    const FwdWs wl = fwd_ws_layout(p.B, p.D, N, pmax);
    p.hsum = static_cast<float*>(ws);
    p.dsum = reinterpret_cast<float*>(static_cast<char*>(ws) + wl.off_dsum);
    p.hin = reinterpret_cast<float*>(static_cast<char*>(ws) + wl.off_hin);
  }
  if (p.P > 1) {
    auto skern = scan_fwd_kernel<N, T, FUSE, true>;
    if (cudaFuncSetAttribute(skern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SS_ERR_CUDA;
    cudaFuncSetAttribute(skern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    skern<<<dim3(ndt, p.B * (p.P - 1)), 32, smem, stream>>>(p, tm[0], tm[1], tm[2], tm[3], tm[4]);
    if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
    if (seg_combine<false>(SegCombine{p.A, p.dsum, p.hsum, p.h0, p.hin, p.P, p.D, N, p.P, 1}, p.B, stream) != cudaSuccess)
      return SS_ERR_CUDA;
    kern<<<dim3(ndt, p.B * p.P), 32, smem, stream>>>(p, tm[0], tm[1], tm[2], tm[3], tm[4]);
  } else {
    // every CTA loops over its batch rows: one wave of equal CTAs when the rows do not fit at once
    const int per_sm = resident_ctas(kern, 32, smem);
    if (per_sm < 1) return SS_ERR_CUDA;
    const int gy = balanced_rows(p.B, ndt, (long long)per_sm * device_sm_count());
    kern<<<dim3(ndt, gy), 32, smem, stream>>>(p, tm[0], tm[1], tm[2], tm[3], tm[4]);
  }
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
// One whole sequence summarised: the summary pass over a single segment [0, L) per batch row.
template <int N, typename T, bool FUSE>
int launch_fwd_summary(FwdParams p, const void* x, const void* delta, const void* Bm, cudaStream_t stream) {
  constexpr int e = ActT<T>::kBytes;
  constexpr int DT = GeoW<N>::DT;
  CUtensorMap tm[3];
  const uint64_t adims[3] = {(uint64_t)p.D, (uint64_t)p.L, (uint64_t)p.B};
  const uint64_t astr[2] = {(uint64_t)p.D * e, (uint64_t)p.L * p.D * e};
  const uint32_t abox[3] = {DT, kTT, 1};
  const uint64_t bdims[2] = {(uint64_t)p.L * N, (uint64_t)p.B};
  const uint64_t bstr[1] = {(uint64_t)p.L * N * e};
  const uint32_t bbox[2] = {kTT * N, 1};
  if (!ssh::encode_tiled(&tm[0], ActT<T>::kTma, 3, delta, adims, astr, abox) ||
      !ssh::encode_tiled(&tm[1], ActT<T>::kTma, 3, x, adims, astr, abox) ||
      !ssh::encode_tiled(&tm[2], ActT<T>::kTma, 2, Bm, bdims, bstr, bbox))
    return SS_ERR_CUDA;
  const size_t smem = sizeof(FwdSmem<T, N>);
  auto skern = scan_fwd_kernel<N, T, FUSE, true>;
  if (cudaFuncSetAttribute(skern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return SS_ERR_CUDA;
  cudaFuncSetAttribute(skern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  p.P = 2;  // one summarised segment per batch row
  p.Ls = p.L;
  p.sum_stride = 1;
  skern<<<dim3((p.D + DT - 1) / DT, p.B), 32, smem, stream>>>(p, tm[0], tm[1], tm[1], tm[2], tm[2]);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <int N, typename T>
int fwd_summary_fuse(const FwdParams& p, const void* x, const void* delta, const void* Bm, cudaStream_t s) {
  return p.fuse ? launch_fwd_summary<N, T, true>(p, x, delta, Bm, s) : launch_fwd_summary<N, T, false>(p, x, delta, Bm, s);
}

}  // namespace

namespace ssh {
int read_clear_fwd_err(cudaStream_t s, unsigned* out) {
  unsigned zero = 0;
  if (cudaMemcpyFromSymbolAsync(out, g_fwd_err, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SS_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_fwd_err, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, s) != cudaSuccess) return SS_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
}  // namespace ssh

namespace {
// the discretisation of delta is a template switch, so the plain scan carries none of it
template <int N, typename T>
int fwd_fuse(const FwdParams& p, const void* x, const void* delta, const void* Bm, const void* Cm, const void* z, void* ws,
             cudaStream_t s) {
  return p.fuse ? launch_fwd<N, T, true>(p, x, delta, Bm, Cm, z, ws, s) : launch_fwd<N, T, false>(p, x, delta, Bm, Cm, z, ws, s);
}
}  // namespace

extern "C" int ss_scan_num_chunks(int L, int chunk) { return (L > 0 && chunk > 0) ? (L + chunk - 1) / chunk : 0; }

namespace {
int validate_fwd(int B, int L, int D, int N, int chunk, int dtype) {
  if (B <= 0 || L <= 0 || D <= 0 || N <= 0 || chunk <= 0) return SS_ERR_DIM;
  if (N != 4 && N != 8 && N != 16) return SS_ERR_UNSUPPORTED;
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if (chunk != kS && chunk % kTT != 0) return SS_ERR_UNSUPPORTED;
  if (D % 8 != 0) return SS_ERR_ALIGN;
  // the B_t / C_t rows of one batch element must span a multiple of 16 bytes (TMA stride rule)
  if (((long long)L * N * (dtype == SS_F32 ? 4 : 2)) % 16 != 0) return SS_ERR_ALIGN;
  // TMA coordinates and tensor extents are 32-bit
  if ((long long)L * N >= (1ll << 31) || (long long)L * D >= (1ll << 40)) return SS_ERR_DIM;
  return SS_OK;
}

}  // namespace

extern "C" size_t ss_scan_fwd_workspace_size(int B, int L, int D, int N, int chunk, int dtype) {
  if (validate_fwd(B, L, D, N, chunk, dtype) != SS_OK) return 0;
  return fwd_ws_bytes(B, L, D, N);
}

extern "C" int ss_scan_fwd(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm, const float* Dv,
                           const void* z, const float* h0, void* y, float* ckpt, float* h_last, int B, int L, int D, int N,
                           int chunk, int dtype, const float* dt_bias, int delta_softplus, void* workspace,
                           size_t ws_bytes, void* stream) {
  if (!x || !delta || !A || !Bm || !Cm || !Dv || !z || !y || !ckpt) return SS_ERR_NULL;
  const int v = validate_fwd(B, L, D, N, chunk, dtype);
  if (v != SS_OK) return v;
  const void* ptrs[] = {x, delta, A, Bm, Cm, Dv, z, y, ckpt};
  for (const void* q : ptrs)
    if (!ssh::aligned16(q)) return SS_ERR_ALIGN;
  if ((h0 && !ssh::aligned16(h0)) || (h_last && !ssh::aligned16(h_last))) return SS_ERR_ALIGN;
  const size_t need = fwd_ws_bytes(B, L, D, N);
  if (need > 0 && (workspace == nullptr || ws_bytes < need)) return SS_ERR_WORKSPACE;
  if (workspace != nullptr && !ssh::aligned16(workspace)) return SS_ERR_ALIGN;
  FwdParams p{A, Dv, h0, y, ckpt, h_last, B, L, D, chunk, ss_scan_num_chunks(L, chunk), 1, L, nullptr, nullptr, nullptr, 1,
              dt_bias, delta_softplus ? 1 : 0, (dt_bias != nullptr || delta_softplus) ? 1 : 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SS_F32) {
    if (N == 4) return fwd_fuse<4, float>(p, x, delta, Bm, Cm, z, workspace, s);
    if (N == 8) return fwd_fuse<8, float>(p, x, delta, Bm, Cm, z, workspace, s);
    return fwd_fuse<16, float>(p, x, delta, Bm, Cm, z, workspace, s);
  }
  if (N == 4) return fwd_fuse<4, __nv_bfloat16>(p, x, delta, Bm, Cm, z, workspace, s);
  if (N == 8) return fwd_fuse<8, __nv_bfloat16>(p, x, delta, Bm, Cm, z, workspace, s);
  return fwd_fuse<16, __nv_bfloat16>(p, x, delta, Bm, Cm, z, workspace, s);
}

extern "C" int ss_scan_fwd_summary(const void* x, const void* delta, const float* A, const void* Bm, float* h_end,
                                   float* delta_sum, int B, int L, int D, int N, int dtype, const float* dt_bias,
                                   int delta_softplus, void* stream) {
  if (!x || !delta || !A || !Bm || !h_end || !delta_sum) return SS_ERR_NULL;
  const int v = validate_fwd(B, L, D, N, kTT, dtype);
  if (v != SS_OK) return v;
  const void* ptrs[] = {x, delta, A, Bm, h_end, delta_sum};
  for (const void* q : ptrs)
    if (!ssh::aligned16(q)) return SS_ERR_ALIGN;
  FwdParams p{A, nullptr, nullptr, nullptr, nullptr, nullptr, B, L, D, kTT, 0, 2, L, h_end, delta_sum, nullptr, 1,
              dt_bias, delta_softplus ? 1 : 0, (dt_bias != nullptr || delta_softplus) ? 1 : 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SS_F32) {
    if (N == 4) return fwd_summary_fuse<4, float>(p, x, delta, Bm, s);
    if (N == 8) return fwd_summary_fuse<8, float>(p, x, delta, Bm, s);
    return fwd_summary_fuse<16, float>(p, x, delta, Bm, s);
  }
  if (N == 4) return fwd_summary_fuse<4, __nv_bfloat16>(p, x, delta, Bm, s);
  if (N == 8) return fwd_summary_fuse<8, __nv_bfloat16>(p, x, delta, Bm, s);
  return fwd_summary_fuse<16, __nv_bfloat16>(p, x, delta, Bm, s);
}

extern "C" int ss_scan_carries(const float* A, const float* delta_sum, const float* summ, const float* init, float* carry,
                               int P, int B, int D, int N, int reverse, void* stream) {
  if (!A || !delta_sum || !summ || !carry) return SS_ERR_NULL;
  if (B <= 0 || P <= 0 || D <= 0 || N <= 0) return SS_ERR_DIM;
  if (P > kSegMax) return SS_ERR_UNSUPPORTED;
  if ((long long)D * N >= (1ll << 31) || B >= 65536) return SS_ERR_DIM;
  const SegCombine c{A, delta_sum, summ, init, carry, P, D, N, 1, B};  // segment-major [P][B]
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = reverse ? seg_combine<true>(c, B, s) : seg_combine<false>(c, B, s);
  return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
