// Selective-scan backward (ss_scan_bwd) for sm_103a: backpropagation through
// time through the diagonal SSM state, with the states rebuilt from the
// forward's chunk checkpoints instead of a stored [B, L, D, N] history.
//
// One CTA = 32 channels (64 when N = 4, or when a chunk's parked states take
// 128 TMEM columns or more) of one batch row at a time.  Chunks are visited from
// last to first; each chunk (a multiple of 16 steps) is walked twice:
//   pass A (tiles in order):   from the chunk's checkpoint, advance
//       h_t = a_t h_{t-1} + delta_t B_t x_t and park the state entering every
//       8-step window in tensor memory (TMEM: each thread owns one TMEM lane);
//   pass B (tiles in reverse): per 8-step window, rebuild a_t and h_t from the
//       parked state into registers (one ex2 per cell), then run the adjoint
//       G_t = ds_t C_t + a_{t+1} G_{t+1} backwards through the window:
//         q_t = (a_t G_t) h_{t-1};  sum_n q_t A  and  sum_n G_t B_t  (-> ddelta, dx)
//         dA += q_t delta_t;  dB_t += G_t delta_t x_t;  dC_t += ds_t h_t.
//       The carry a_t G_t crosses windows, tiles and chunks in registers.
// With chunk = 8 every window has its own checkpoint and pass A is skipped.
// Inside the step loops every thread only adds its own cells and stores its
// shares to shared memory; the window epilogue adds the shares in a fixed
// order (over the 4-state lane groups for the per-(t,d) sums, over lanes and
// warps for dB_t, dC_t) and writes dx, ddelta, dz and one dB/dC partial per
// channel tile.  ss_bwd_reduce_kernel adds the partials of
// dB/dC and of dA/dD in fixed order.  No atomics: results are bitwise
// reproducible.
// Sequence segments (few batch rows, long sequences): a summary kernel gives
// each later segment's adjoint at its start from a zero carry and its sum of
// delta; the warp-shuffle associative scan of scan_common.cuh composes them
// into the carry arriving at the end of every segment, from which each
// segment's CTAs run independently.
#include "scan_common.cuh"

namespace {

using namespace ssk;

__device__ unsigned g_bwd_err;

// Channels per CTA: 32 (two warps at N = 16) so that a Mamba-sized layer has
// enough CTAs to keep ~4 per SM; N = 4 needs 64 (one warp spans 64 channels).
template <int N>
constexpr int bwd_dt() {
  return Geo<N, 64>::WC > 32 ? 64 : 32;
}

// Window groups of a backward CTA: two when a 64-channel CTA has four warps (N = 16), else one.
__host__ __device__ constexpr int bwd_groups(int N, int DT) {
  return (DT == 64 && N == 16) ? 2 : 1;
}

template <typename T, int N, int NSTG, int DT>
struct BwdSmem {
  static constexpr int W = Geo<N, DT>::W, CG = Geo<N, DT>::CG;
  static constexpr int kSP = DT + 8;       // row pitch of the C.h shares (bank spread across lane groups)
  static constexpr int kSAB = 2 * DT + 8;  // row pitch of the (sum qA, sum GB) shares
  alignas(128) T dlt[NSTG][kTT * DT];
  alignas(128) T x[NSTG][kTT * DT];
  alignas(128) T z[NSTG][kTT * DT];
  alignas(128) T dy[NSTG][kTT * DT];
  alignas(128) T Bm[NSTG][kTT * N];
  alignas(128) T Cm[NSTG][kTT * N];
  alignas(16) float dlt_f[kTT * DT];
  alignas(16) float dx_f[kTT * DT];  // delta * x
  alignas(16) float ds_f[kTT * DT];  // dy * silu(z)
  alignas(16) float x_f[kTT * DT];   // x
  alignas(16) float gz_f[kTT * DT];  // dy * silu'(z) = dy * sig(z) * (1 + z (1 - sig(z)))
  alignas(16) float B_f[kTT * N];
  alignas(16) float C_f[kTT * N];
  // one 8-step window's per-lane shares
  alignas(16) float sp[kS][N / 4][kSP];    // C_t . h_t over the lane's 4 states
  alignas(16) float sab[kS][N / 4][kSAB];  // (sum q A log2 e, sum G B) over the lane's 4 states, per channel
  // [warp][step][dB | dC][channel-pair group x state]: G_t delta_t x_t and ds_t h_t summed over
  // the lane's 2 channels (row pitch CG*N + 16 keeps the epilogue's 128-bit reads conflict-free)
  alignas(16) float dbc[W][kS][2][CG * N + 16];
  alignas(16) float Dv_s[DT];
  alignas(16) float bias_s[DT];  // dt_bias of the fused discretisation (0 without one)
  alignas(8) uint64_t full[NSTG];
  uint32_t tmem_base;
};

// Four 32-channel bf16 CTAs (N = 16, the register-limited residency) must also
// fit the SM's 228 KB of shared memory, 1 KB of which each CTA reserves.
static_assert(sizeof(BwdSmem<__nv_bfloat16, 16, 1, 32>) + 1024 <= 228 * 1024 / 4, "four backward CTAs per SM");

// TMEM columns: 8 per window boundary of a chunk, rounded up to a power of two >= 32
inline uint32_t tmem_cols(int chunk) {
  uint32_t need = (uint32_t)(chunk / kS) * 8u, c = 32;
  while (c < need) c <<= 1;
  return c;
}
constexpr int kMaxChunk = 512;  // 64 windows x 8 columns = the 512 TMEM columns of an SM

struct BwdParams {
  const float* A;
  const float* Dv;
  const float* ckpt;
  const float* dh_last;
  float* dx;
  float* ddelta;
  float* dz;
  float* dh0;
  float* ws_dBC;  // [channel tiles x window groups][B][L][2N]
  float* ws_dAD;  // [CTA rows][D*N + 2D]: dA, dD and d dt_bias partials of each CTA row
  int B, L, D, chunk, nchunks;
  uint32_t tcols;
  int P, Ls;      // sequence segments (P = 1: one CTA row walks whole batch rows)
  float* gsum;    // [B][P][D][N] adjoint a_tb G_tb at each segment's start from a zero carry at its end
  float* dsum;    // [B][P][D]    sum of delta over each segment
  float* gin;     // [B][P][D][N] carry a G arriving at the end of each segment (combine kernel output)
  int sum_stride, sum_first;  // summary grid: rows per batch row and first segment (P and 1 inside ss_scan_bwd)
  const float* dt_bias;  // fused discretisation: delta = f(raw + dt_bias), f = softplus if dsp
  int dsp;
  int fuse;              // dt_bias != NULL or dsp
  float* d_dt_bias;      // [D] accumulated gradient of dt_bias, or NULL
};

template <typename T, int N, int NSTG, int DT>
struct BwdSumSmem {
  alignas(128) T dlt[NSTG][kTT * DT];
  alignas(128) T z[NSTG][kTT * DT];
  alignas(128) T dy[NSTG][kTT * DT];
  alignas(128) T Cm[NSTG][kTT * N];
  alignas(16) float dlt_f[kTT * DT];
  alignas(16) float ds_f[kTT * DT];
  alignas(16) float C_f[kTT * N];
  alignas(16) float bias_s[DT];
  alignas(8) uint64_t full[NSTG];
};

// Summary-kernel geometry: one channel x 4 states per thread (the summary keeps
// no per-step shares, so its threads can be half as wide as the main kernel's
// and the segments get twice the warps), lane = ng * CPW + c so that the lanes
// reading one state quad of C_t are consecutive.
template <int N, int DT>
struct GeoS {
  static constexpr int NG = N / 4;      // lanes per channel
  static constexpr int CPW = 32 / NG;   // channels per warp
  static constexpr int W = DT / CPW;    // warps per CTA
  static constexpr int NT = 32 * W;
  static_assert(W >= 1 && DT % CPW == 0, "a CTA holds whole warps");
};

// Channels per summary CTA: one warp's worth.  A one-warp CTA's tile barrier
// costs nothing, where eight-warp CTAs stalled on it (long-context backward
// 1006 -> 964 us, with four staging slots instead of six so that the narrower
// CTAs, which share less of the B_t/C_t staging, still all fit at once).
template <int N>
constexpr int sum_dt() {
  return GeoS<N, 32 / (N / 4)>::CPW;
}

// Segment summaries: for each segment the adjoint it carries out of its first
// step when the carry entering its last step is zero, and its sum of delta.
// CTA = (channel tile, (batch row, segment)); tiles walked last to first.
template <int N, typename T, int NSTG, int DT, bool FUSE>
__global__ void __launch_bounds__(GeoS<N, DT>::NT) scan_bwd_summary_kernel(const BwdParams p,
                                                                        const __grid_constant__ CUtensorMap tm_dlt,
                                                                        const __grid_constant__ CUtensorMap tm_z,
                                                                        const __grid_constant__ CUtensorMap tm_dy,
                                                                        const __grid_constant__ CUtensorMap tm_C) {
  using G = GeoS<N, DT>;
  using AT = ActT<T>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  BwdSumSmem<T, N, NSTG, DT>& S = *reinterpret_cast<BwdSumSmem<T, N, NSTG, DT>*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ng = lane / G::CPW, c = lane % G::CPW;
  const int dl = warp * G::CPW + c;
  const int d0 = blockIdx.x * DT;
  const int dg = d0 + dl;
  const bool dvalid = dg < p.D;
  const int n0 = ng * 4;
  const int b = (int)blockIdx.y / (p.P - 1), sgm = p.sum_first + (int)blockIdx.y % (p.P - 1);
  const int tb = sgm * p.Ls, te = min(p.L, tb + p.Ls);
  const int gtb = tb / kTT, gte = (te + kTT - 1) / kTT;
  const int nitems = gte - gtb;
  constexpr uint32_t kActBytes = kTT * DT * AT::kBytes;
  constexpr uint32_t kStageBytes = 3 * kActBytes + kTT * N * AT::kBytes;
  float2 Ap[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float* a = p.A + (size_t)(dvalid ? dg : 0) * N + n0 + 2 * q;
    Ap[q] = dvalid ? f2(a[0] * kLog2e, a[1] * kLog2e) : f2(0.f, 0.f);
  }
  auto issue = [&](int k) {
    fence_proxy_async_smem();  // the slot's earlier readers passed a barrier before this call
    const int slot = k % NSTG, t0 = (gte - 1 - k) * kTT;
    mbar_arrive_expect_tx(&S.full[slot], kStageBytes);
    tma_load_3d(S.dlt[slot], &tm_dlt, &S.full[slot], d0, t0, b);
    tma_load_3d(S.z[slot], &tm_z, &S.full[slot], d0, t0, b);
    tma_load_3d(S.dy[slot], &tm_dy, &S.full[slot], d0, t0, b);
    tma_load_2d(S.Cm[slot], &tm_C, &S.full[slot], t0 * N, b);
  };
  for (int cc = tid; cc < DT; cc += G::NT) S.bias_s[cc] = (p.dt_bias != nullptr && d0 + cc < p.D) ? p.dt_bias[d0 + cc] : 0.f;
  if (tid == 0) {
    prefetch_tmap(&tm_dlt); prefetch_tmap(&tm_z); prefetch_tmap(&tm_dy); prefetch_tmap(&tm_C);
    for (int st = 0; st < NSTG; ++st) mbar_init(&S.full[st], 1);
    fence_barrier_init();
    for (int k = 0; k < NSTG && k < nitems; ++k) issue(k);
  }
  __syncthreads();
  float2 ga[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
  float dsum = 0.f;
  for (int k = 0; k < nitems; ++k) {
    const int slot = k % NSTG;
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
    for (int gi = tid; gi < kTT * DT / 4; gi += G::NT) {
      float dv[4], zv[4], gv[4];
      AT::ld4(&S.dlt[slot][gi * 4], dv);
      AT::ld4(&S.z[slot][gi * 4], zv);
      AT::ld4(&S.dy[slot][gi * 4], gv);
      if constexpr (FUSE) {
        const int c4 = (gi % (DT / 4)) * 4;
        delta_transform4(dv, S.bias_s, c4, (gte - 1 - k) * kTT + gi / (DT / 4) < p.L, p.D - d0 - c4, p.dsp);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) gv[e] *= zv[e] * sigmoid(zv[e]);
      reinterpret_cast<float4*>(S.dlt_f)[gi] = make_float4(dv[0], dv[1], dv[2], dv[3]);
      reinterpret_cast<float4*>(S.ds_f)[gi] = make_float4(gv[0], gv[1], gv[2], gv[3]);
    }
    for (int gi = tid; gi < kTT * N / 4; gi += G::NT) {
      float cv[4];
      AT::ld4(&S.Cm[slot][gi * 4], cv);
      reinterpret_cast<float4*>(S.C_f)[gi] = make_float4(cv[0], cv[1], cv[2], cv[3]);
    }
    __syncthreads();
    if (tid == 0 && k + NSTG < nitems) issue(k + NSTG);  // the slot is widened: refill it
#pragma unroll
    for (int r = kTT - 1; r >= 0; --r) {
      const float dj = S.dlt_f[r * DT + dl];
      const float2 gj = bc2(S.ds_f[r * DT + dl]);
      const float4 Cv = *reinterpret_cast<const float4*>(&S.C_f[r * N + n0]);
      const float2 d2 = bc2(dj);
      dsum += dj;
      ga[0] = mul2(ex2_2(mul2(d2, Ap[0])), fma2(gj, f2(Cv.x, Cv.y), ga[0]));
      ga[1] = mul2(ex2_2(mul2(d2, Ap[1])), fma2(gj, f2(Cv.z, Cv.w), ga[1]));
    }
    __syncthreads();
  }
  if (dvalid) {
    const size_t row = ((size_t)b * p.sum_stride + sgm) * p.D + dg;
    *reinterpret_cast<float4*>(p.gsum + row * N + n0) = make_float4(ga[0].x, ga[0].y, ga[1].x, ga[1].y);
    if (ng == 0) p.dsum[row] = dsum;
  }
}

template <int N, typename T, int NSTG, int DT, bool FUSE>
__global__ void __launch_bounds__(Geo<N, DT>::NT) scan_bwd_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tm_dlt,
                                                              const __grid_constant__ CUtensorMap tm_x,
                                                              const __grid_constant__ CUtensorMap tm_z,
                                                              const __grid_constant__ CUtensorMap tm_dy,
                                                              const __grid_constant__ CUtensorMap tm_B,
                                                              const __grid_constant__ CUtensorMap tm_C) {
  using G = Geo<N, DT>;
  using AT = ActT<T>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  BwdSmem<T, N, NSTG, DT>& S = *reinterpret_cast<BwdSmem<T, N, NSTG, DT>*>(smem_raw);

  pdl_trigger();  // the reduction of the partials may launch now; it waits for this grid's end
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ng = lane % G::NG, cg = lane / G::NG;
  const int dl = warp * G::WC + cg * 2;
  const int d0 = blockIdx.x * DT;
  const int dg = d0 + dl;
  const bool dvalid = dg < p.D;
  const int n0 = ng * 4;
  const int L = p.L;
  // P = 1: CTA row y walks batch rows y, y + gridDim.y, ... whole.
  // P > 1: CTA row y owns one segment [tb, te) of batch row y / P; segments are
  // whole chunks and whole tiles, so only the last one can be ragged.
  const bool segs = p.P > 1;
  const int sgm = segs ? (int)blockIdx.y % p.P : 0;
  const int tb = sgm * p.Ls, te = segs ? min(L, tb + p.Ls) : L;
  const int gtb = tb / kTT, gte = (te + kTT - 1) / kTT;  // tiles [gtb, gte)
  const int ntiles = gte - gtb;
  const bool direct = p.chunk == kS;                    // a checkpoint per window: no pass A
  const int tpc = direct ? 1 : p.chunk / kTT;           // tiles per full chunk
  const int ce = direct ? 0 : (te + p.chunk - 1) / p.chunk;  // chunks [tb / chunk, ce)
  const int ntl = gte - (ce - 1) * tpc;                 // tiles in the segment's last chunk
  const int per_b = direct ? ntiles : 2 * ntiles;       // items per batch row
  const int nb = segs ? 1 : (p.B - (int)blockIdx.y + (int)gridDim.y - 1) / (int)gridDim.y;
  const int nitems = nb * per_b;
  constexpr uint32_t kActBytes = kTT * DT * AT::kBytes;
  constexpr uint32_t kBCBytes = kTT * N * AT::kBytes;
  // A four-warp CTA (64 channels, so that the TMEM of a long chunk is used on
  // all 128 lanes) closes its windows as two 32-channel groups of two warps,
  // each with its own barrier and its own dB/dC partial: a window then waits
  // for one other warp instead of three.  Tiles (staging, widening) stay CTA-wide.
  constexpr int GRP = bwd_groups(N, DT);
  constexpr int GT = G::NT / GRP, GW = G::W / GRP, GDT = DT / GRP;
  const int grp = warp / GW, gtid = tid - grp * GT;
  auto group_sync = [&]() {
    if constexpr (GRP == 1) __syncthreads();
    else asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(GT) : "memory");
  };

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
  for (int c = tid; c < DT; c += G::NT) {
    S.Dv_s[c] = (d0 + c < p.D) ? p.Dv[d0 + c] : 0.f;
    S.bias_s[c] = (p.dt_bias != nullptr && d0 + c < p.D) ? p.dt_bias[d0 + c] : 0.f;
  }

  // Items of a batch row, in order.  Direct mode: tiles gte-1 down to gtb.
  // Otherwise per chunk kc = ce-1 down to tb/chunk: pass A over its ntc tiles
  // in order, then pass B over them in reverse.  Two cursors (consumer, TMA
  // issuer) step through the items without divisions.
  const int kc_first = tb / p.chunk;
  struct Cursor {
    int b, kc, tl, ntc;
    bool passB, first;
  };
  auto start_row = [&](Cursor& c, int b) {
    c.b = b;
    c.first = true;
    if (direct) {
      c.kc = gte - 1;  // the tile
      c.tl = 0;
      c.ntc = 1;
      c.passB = true;
    } else {
      c.kc = ce - 1;
      c.ntc = ntl;
      c.tl = 0;
      c.passB = false;
    }
  };
  auto advance = [&](Cursor& c) {
    c.first = false;
    if (direct) {
      if (--c.kc < gtb) start_row(c, c.b + (int)gridDim.y);
      return;
    }
    if (!c.passB) {
      if (++c.tl == c.ntc) {
        c.passB = true;
        c.tl = c.ntc - 1;
      }
    } else if (c.tl-- == 0) {
      if (--c.kc < kc_first) {
        start_row(c, c.b + (int)gridDim.y);
      } else {
        c.ntc = tpc;
        c.tl = 0;
        c.passB = false;
      }
    }
  };
  auto tile_of = [&](const Cursor& c) { return direct ? c.kc : c.kc * tpc + c.tl; };
  const int b_first = segs ? (int)blockIdx.y / p.P : (int)blockIdx.y;
  Cursor icur;
  start_row(icur, b_first);
  auto issue = [&](int k) {  // k: the item icur points at
    fence_proxy_async_smem();  // the slot's earlier readers passed a barrier before this call
    const int b = icur.b, gt = tile_of(icur);
    const bool passB = icur.passB;
    advance(icur);
    const int slot = k % NSTG;
    const int t0 = gt * kTT;
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

  if (warp == 0) {
    if (!direct) tmem_alloc(&S.tmem_base, p.tcols);
    tmem_relinquish();
  }
  if (tid == 0) {
    prefetch_tmap(&tm_dlt); prefetch_tmap(&tm_x); prefetch_tmap(&tm_z);
    prefetch_tmap(&tm_dy); prefetch_tmap(&tm_B); prefetch_tmap(&tm_C);
    for (int s = 0; s < NSTG; ++s) mbar_init(&S.full[s], 1);
    fence_barrier_init();
    for (int k = 0; k < NSTG && k < nitems; ++k) issue(k);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // this thread's TMEM lane: 32 * (warp % 4) + lane; window boundary sb at columns [8 sb, 8 sb + 8)
  const uint32_t tlane = direct ? 0u : S.tmem_base + ((uint32_t)(32 * (warp & 3)) << 16);

  float2 h[2][2];              // pass-A running state
  float2 ga[2][2];             // a_{t+1} * G_{t+1}: the adjoint carried backwards
  float2 dA2[2][2];            // dA partial sums of the thread's cells
  float dDacc[4];              // dD partial sums of the epilogue's four channels
  float dTacc[4];              // d dt_bias partial sums of the same channels
#pragma unroll
  for (int j = 0; j < 2; ++j) dA2[j][0] = dA2[j][1] = f2(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < 4; ++e) dDacc[e] = dTacc[e] = 0.f;
  bool failed = false;

  Cursor cur;
  start_row(cur, b_first);
  for (int k = 0; k < nitems; ++k, advance(cur)) {
    const int slot = k % NSTG;
    const int b = cur.b;
    const int gt = tile_of(cur);
    const bool passB = cur.passB;
    const bool lastA = !cur.passB && cur.tl == cur.ntc - 1;  // last pass-A tile of its chunk
    const int t0 = gt * kTT;
    const int kc = cur.kc, tl = cur.tl;

    if (cur.first) {  // entering batch row b: the gradient arriving on h_{te-1}
      // (with segments, the combine kernel composed it from dh_last and the later segments' summaries)
      const float* src = segs ? p.gin + ((size_t)b * p.P + sgm) * p.D * N
                              : (p.dh_last ? p.dh_last + (size_t)b * p.D * N : nullptr);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src != nullptr && dvalid) v = *reinterpret_cast<const float4*>(src + (size_t)(dg + j) * N + n0);
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
      failed = true;
      break;
    }

    if (!passB) {
      // ------------------------------------------------ pass A: park window states
      if (tl == 0) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (dvalid) v = *reinterpret_cast<const float4*>(p.ckpt + (((size_t)b * p.nchunks + kc) * p.D + dg + j) * N + n0);
          h[j][0] = f2(v.x, v.y);
          h[j][1] = f2(v.z, v.w);
        }
      }
      for (int gi = tid; gi < kTT * DT / 4; gi += G::NT) {
        float dv[4], xv[4];
        AT::ld4(&S.dlt[slot][gi * 4], dv);
        AT::ld4(&S.x[slot][gi * 4], xv);
        if constexpr (FUSE) {
          const int c4 = (gi % (DT / 4)) * 4;
          delta_transform4(dv, S.bias_s, c4, t0 + gi / (DT / 4) < L, p.D - d0 - c4, p.dsp);
        }
        reinterpret_cast<float4*>(S.dlt_f)[gi] = make_float4(dv[0], dv[1], dv[2], dv[3]);
        reinterpret_cast<float4*>(S.dx_f)[gi] = make_float4(dv[0] * xv[0], dv[1] * xv[1], dv[2] * xv[2], dv[3] * xv[3]);
      }
      for (int gi = tid; gi < kTT * N / 4; gi += G::NT) {
        float bv[4];
        AT::ld4(&S.Bm[slot][gi * 4], bv);
        reinterpret_cast<float4*>(S.B_f)[gi] = make_float4(bv[0], bv[1], bv[2], bv[3]);
      }
      __syncthreads();
      if (tid == 0 && k + NSTG < nitems) issue(k + NSTG);
#pragma unroll
      for (int half = 0; half < kTT / kS; ++half) {
        tmem_st8(tlane + (uint32_t)((tl * (kTT / kS) + half) * 8),
                 make_float4(h[0][0].x, h[0][0].y, h[0][1].x, h[0][1].y),
                 make_float4(h[1][0].x, h[1][0].y, h[1][1].x, h[1][1].y));
        float2 av[kS][2][2];
#pragma unroll
        for (int i = 0; i < kS; ++i) {  // exponentials first: independent of the state
          const float2 dd = *reinterpret_cast<const float2*>(&S.dlt_f[(half * kS + i) * DT + dl]);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float2 dj = bc2(j ? dd.y : dd.x);
            av[i][j][0] = ex2_2(mul2(dj, Ap[j][0]));
            av[i][j][1] = ex2_2(mul2(dj, Ap[j][1]));
          }
        }
#pragma unroll
        for (int i = 0; i < kS; ++i) {
          const int r = half * kS + i;
          const float2 xx = *reinterpret_cast<const float2*>(&S.dx_f[r * DT + dl]);
          const float4 Bv = *reinterpret_cast<const float4*>(&S.B_f[r * N + n0]);
          const float2 B01 = f2(Bv.x, Bv.y), B23 = f2(Bv.z, Bv.w);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float2 xj = bc2(j ? xx.y : xx.x);
            h[j][0] = fma2(av[i][j][0], h[j][0], mul2(xj, B01));
            h[j][1] = fma2(av[i][j][1], h[j][1], mul2(xj, B23));
          }
        }
      }
      if (lastA) tmem_wait_st();  // the chunk's states are parked before pass B reads them
      __syncthreads();
      continue;
    }

    // -------------------------------------------------- pass B: adjoint sweep
    float4 hck[kTT / kS][2];  // direct mode: the checkpoints entering the tile's two windows
    if (direct) {
#pragma unroll
      for (int w = 0; w < kTT / kS; ++w)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = gt * (kTT / kS) + w;
          hck[w][j] = (dvalid && c < p.nchunks)
                          ? *reinterpret_cast<const float4*>(p.ckpt + (((size_t)b * p.nchunks + c) * p.D + dg + j) * N + n0)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // widen the tile once: everything the windows and their epilogues read is
    // fp32 in shared memory, so the staging slot is free after this pass
    for (int gi = tid; gi < kTT * DT / 4; gi += G::NT) {
      float dv[4], xv[4], zv[4], gv[4], dxv[4], dsv[4], gzv[4];
      AT::ld4(&S.dlt[slot][gi * 4], dv);
      AT::ld4(&S.x[slot][gi * 4], xv);
      AT::ld4(&S.z[slot][gi * 4], zv);
      AT::ld4(&S.dy[slot][gi * 4], gv);
      if constexpr (FUSE) {
        const int c4 = (gi % (DT / 4)) * 4;
        delta_transform4(dv, S.bias_s, c4, t0 + gi / (DT / 4) < L, p.D - d0 - c4, p.dsp);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float sg = sigmoid(zv[e]);
        dxv[e] = xv[e] * dv[e];
        dsv[e] = gv[e] * (zv[e] * sg);
        gzv[e] = gv[e] * sg * fmaf(zv[e], 1.0f - sg, 1.0f);
      }
      reinterpret_cast<float4*>(S.dlt_f)[gi] = make_float4(dv[0], dv[1], dv[2], dv[3]);
      reinterpret_cast<float4*>(S.dx_f)[gi] = make_float4(dxv[0], dxv[1], dxv[2], dxv[3]);
      reinterpret_cast<float4*>(S.ds_f)[gi] = make_float4(dsv[0], dsv[1], dsv[2], dsv[3]);
      reinterpret_cast<float4*>(S.x_f)[gi] = make_float4(xv[0], xv[1], xv[2], xv[3]);
      reinterpret_cast<float4*>(S.gz_f)[gi] = make_float4(gzv[0], gzv[1], gzv[2], gzv[3]);
    }
    for (int gi = tid; gi < kTT * N / 4; gi += G::NT) {
      float bv[4], cv[4];
      AT::ld4(&S.Bm[slot][gi * 4], bv);
      AT::ld4(&S.Cm[slot][gi * 4], cv);
      reinterpret_cast<float4*>(S.B_f)[gi] = make_float4(bv[0], bv[1], bv[2], bv[3]);
      reinterpret_cast<float4*>(S.C_f)[gi] = make_float4(cv[0], cv[1], cv[2], cv[3]);
    }
    __syncthreads();
    if (tid == 0 && k + NSTG < nitems) issue(k + NSTG);

    for (int sub = kTT / kS - 1; sub >= 0; --sub) {
      const int sb = tl * (kTT / kS) + sub;
      float2 hb[2][2];
      {
        float4 v0, v1;
        if (direct) {
          v0 = sub ? hck[1][0] : hck[0][0];
          v1 = sub ? hck[1][1] : hck[0][1];
        } else {
          tmem_ld8_wait(tlane + (uint32_t)(sb * 8), v0, v1);
        }
        hb[0][0] = f2(v0.x, v0.y); hb[0][1] = f2(v0.z, v0.w);
        hb[1][0] = f2(v1.x, v1.y); hb[1][1] = f2(v1.z, v1.w);
      }
      float2 av[kS][2][2], hv[kS][2][2];
#pragma unroll
      for (int i = 0; i < kS; ++i) {  // exponentials first: independent of the state
        const float2 dd = *reinterpret_cast<const float2*>(&S.dlt_f[(sub * kS + i) * DT + dl]);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 dj = bc2(j ? dd.y : dd.x);
          av[i][j][0] = ex2_2(mul2(dj, Ap[j][0]));
          av[i][j][1] = ex2_2(mul2(dj, Ap[j][1]));
        }
      }
      // rebuild the window's states; shares of C.h and dC on the way
#pragma unroll
      for (int i = 0; i < kS; ++i) {
        const int r = sub * kS + i;
        const float2 xx = *reinterpret_cast<const float2*>(&S.dx_f[r * DT + dl]);
        const float2 gg = *reinterpret_cast<const float2*>(&S.ds_f[r * DT + dl]);
        const float4 Bv = *reinterpret_cast<const float4*>(&S.B_f[r * N + n0]);
        const float4 Cv = *reinterpret_cast<const float4*>(&S.C_f[r * N + n0]);
        const float2 B01 = f2(Bv.x, Bv.y), B23 = f2(Bv.z, Bv.w);
        const float2 C01 = f2(Cv.x, Cv.y), C23 = f2(Cv.z, Cv.w);
        float yj[2];
        float2 dc0, dc1;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 xj = bc2(j ? xx.y : xx.x);
          const float2 gj = bc2(j ? gg.y : gg.x);
          const float2 hp0 = i ? hv[i - 1][j][0] : hb[j][0];
          const float2 hp1 = i ? hv[i - 1][j][1] : hb[j][1];
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
        *reinterpret_cast<float2*>(&S.sp[i][ng][dl]) = f2(yj[0], yj[1]);
        *reinterpret_cast<float4*>(&S.dbc[warp][i][1][cg * N + n0]) = make_float4(dc0.x, dc0.y, dc1.x, dc1.y);
      }
      // adjoint sweep backwards through the window
#pragma unroll
      for (int i = kS - 1; i >= 0; --i) {
        const int r = sub * kS + i;
        const float2 dd = *reinterpret_cast<const float2*>(&S.dlt_f[r * DT + dl]);
        const float2 xx = *reinterpret_cast<const float2*>(&S.dx_f[r * DT + dl]);
        const float2 gg = *reinterpret_cast<const float2*>(&S.ds_f[r * DT + dl]);
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
        *reinterpret_cast<float4*>(&S.sab[i][ng][2 * dl]) = make_float4(sA[0], sB[0], sA[1], sB[1]);
        *reinterpret_cast<float4*>(&S.dbc[warp][i][0][cg * N + n0]) = make_float4(db0.x, db0.y, db1.x, db1.y);
      }
      group_sync();

      // window epilogue.  dB_t, dC_t of this group's channels: lanes and warps in fixed order
      for (int e = gtid; e < kS * N / 2; e += GT) {  // (row, dB | dC, group of 4 states)
        const int i = e / (N / 2), qq = (e % (N / 2)) / (N / 4), n4 = (e % (N / 4)) * 4;
        const int t = t0 + sub * kS + i;
        float2 a01 = f2(0.f, 0.f), a23 = f2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < GW; ++w)
#pragma unroll
          for (int c = 0; c < G::CG; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(&S.dbc[grp * GW + w][i][qq][c * N + n4]);
            a01 = add2(a01, f2(v.x, v.y));
            a23 = add2(a23, f2(v.z, v.w));
          }
        if (t < L)
          *reinterpret_cast<float4*>(
              &p.ws_dBC[(((size_t)(blockIdx.x * GRP + grp) * p.B + b) * L + t) * (2 * N) + qq * N + n4]) =
              make_float4(a01.x, a01.y, a23.x, a23.y);
      }
      // per-(t, d) gradients of this group's channels, four channels per thread
      for (int gi = gtid; gi < kS * GDT / 4; gi += GT) {
        const int i = gi / (GDT / 4), c4 = grp * GDT + (gi % (GDT / 4)) * 4;
        const int rr = sub * kS + i;
        const int t = t0 + rr, d = d0 + c4;
        if (t < L && d < p.D) {
          float o0[4], o1[4], o2[4];
          const float4 s4 = *reinterpret_cast<const float4*>(&S.sp[i][0][c4]);
          const float4 a4 = *reinterpret_cast<const float4*>(&S.sab[i][0][2 * c4]);
          const float4 b4 = *reinterpret_cast<const float4*>(&S.sab[i][0][2 * c4 + 4]);
          float2 s01 = f2(s4.x, s4.y), s23 = f2(s4.z, s4.w);
          float2 ab00 = f2(a4.x, a4.y), ab01 = f2(a4.z, a4.w), ab10 = f2(b4.x, b4.y), ab11 = f2(b4.z, b4.w);
#pragma unroll
          for (int g = 1; g < N / 4; ++g) {
            const float4 u = *reinterpret_cast<const float4*>(&S.sp[i][g][c4]);
            const float4 v0 = *reinterpret_cast<const float4*>(&S.sab[i][g][2 * c4]);
            const float4 v1 = *reinterpret_cast<const float4*>(&S.sab[i][g][2 * c4 + 4]);
            s01 = add2(s01, f2(u.x, u.y));
            s23 = add2(s23, f2(u.z, u.w));
            ab00 = add2(ab00, f2(v0.x, v0.y));
            ab01 = add2(ab01, f2(v0.z, v0.w));
            ab10 = add2(ab10, f2(v1.x, v1.y));
            ab11 = add2(ab11, f2(v1.z, v1.w));
          }
          const float4 dv4 = *reinterpret_cast<const float4*>(&S.dlt_f[rr * DT + c4]);
          const float4 xv4 = *reinterpret_cast<const float4*>(&S.x_f[rr * DT + c4]);
          const float4 dsv = *reinterpret_cast<const float4*>(&S.ds_f[rr * DT + c4]);
          const float4 gz4 = *reinterpret_cast<const float4*>(&S.gz_f[rr * DT + c4]);
          const float4 Dd4 = *reinterpret_cast<const float4*>(&S.Dv_s[c4]);
          const float shv[4] = {s01.x, s01.y, s23.x, s23.y};
          const float sAv[4] = {ab00.x, ab01.x, ab10.x, ab11.x};
          const float sBv[4] = {ab00.y, ab01.y, ab10.y, ab11.y};
          const float dv[4] = {dv4.x, dv4.y, dv4.z, dv4.w};
          const float xv[4] = {xv4.x, xv4.y, xv4.z, xv4.w};
          const float gz[4] = {gz4.x, gz4.y, gz4.z, gz4.w};
          const float dsa[4] = {dsv.x, dsv.y, dsv.z, dsv.w};
          const float Dd[4] = {Dd4.x, Dd4.y, Dd4.z, Dd4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float s = fmaf(Dd[e], xv[e], shv[e]);
            o0[e] = fmaf(dsa[e], Dd[e], dv[e] * sBv[e]);  // dx
            o1[e] = fmaf(sAv[e], kLn2, xv[e] * sBv[e]);   // ddelta
            o2[e] = gz[e] * s;                             // dz
            dDacc[e] = fmaf(dsa[e], xv[e], dDacc[e]);
          }
          if constexpr (FUSE) {  // back through delta = softplus(v): softplus'(v) = sigmoid(v) = 1 - exp(-delta)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (p.dsp) o1[e] *= softplus_grad_from_delta(dv[e]);
              dTacc[e] += o1[e];
            }
          }
          const size_t off = ((size_t)b * L + t) * p.D + d;
          *reinterpret_cast<float4*>(p.dx + off) = make_float4(o0[0], o0[1], o0[2], o0[3]);
          *reinterpret_cast<float4*>(p.ddelta + off) = make_float4(o1[0], o1[1], o1[2], o1[3]);
          *reinterpret_cast<float4*>(p.dz + off) = make_float4(o2[0], o2[1], o2[2], o2[3]);
        }
      }
      group_sync();
    }

    if (t0 == 0 && p.dh0 != nullptr && dvalid) {  // last item of batch row b: ga = a_0 G_0
#pragma unroll
      for (int j = 0; j < 2; ++j)
        *reinterpret_cast<float4*>(p.dh0 + ((size_t)b * p.D + dg + j) * N + n0) =
            make_float4(ga[j][0].x, ga[j][0].y, ga[j][1].x, ga[j][1].y);
    }
  }

  // release the tensor memory (every warp is past its last TMEM access)
  if (!direct) tmem_wait_st();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0 && !direct) tmem_dealloc(S.tmem_base, p.tcols);
  if (failed) {  // a CTA that gave up on a wait adds nothing to the accumulated gradients
#pragma unroll
    for (int j = 0; j < 2; ++j) dA2[j][0] = dA2[j][1] = f2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < 4; ++e) dDacc[e] = dTacc[e] = 0.f;
  }

  // per-CTA partials of dA, dD and d dt_bias (summed over this CTA's batch rows)
  float* row = p.ws_dAD + (size_t)blockIdx.y * p.D * (N + 2);
  if (dvalid) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      *reinterpret_cast<float4*>(row + (size_t)(dg + j) * N + n0) =
          make_float4(dA2[j][0].x, dA2[j][0].y, dA2[j][1].x, dA2[j][1].y);
  }
  // dD, d dt_bias: the threads of a group with equal gtid % (GDT/4) hold the same four channels
  float* red = &S.sab[0][0][0];  // free after the last window
  *reinterpret_cast<float4*>(&red[tid * 4]) = make_float4(dDacc[0], dDacc[1], dDacc[2], dDacc[3]);
  *reinterpret_cast<float4*>(&red[(G::NT + tid) * 4]) = make_float4(dTacc[0], dTacc[1], dTacc[2], dTacc[3]);
  __syncthreads();
  for (int c = tid; c < DT; c += G::NT) {
    if (d0 + c < p.D) {
      const int g0 = c / GDT, q4 = (c % GDT) / 4, e = c % 4;
      float accD = 0.f, accT = 0.f;
      for (int m = g0 * GT + q4; m < (g0 + 1) * GT; m += GDT / 4) {
        accD += red[m * 4 + e];
        accT += red[(G::NT + m) * 4 + e];
      }
      row[(size_t)p.D * N + d0 + c] = accD;
      row[(size_t)p.D * (N + 1) + d0 + c] = accT;
    }
  }
}

// dA (first D*N columns of a partial row), dD (next D) and d dt_bias (last D,
// when asked for) accumulate.
struct DADStore {
  float* dA;
  float* dD;
  float* dT;
  long long nA, D;
  __device__ void put(long long i, float v) const {
    if (i < nA) dA[i] += v;
    else if (i < nA + D) dD[i - nA] += v;
    else if (dT != nullptr) dT[i - nA - D] += v;
  }
};

// The backward's fixed-order reductions in one launch.  Blocks [0, nblk_bc):
// dB, dC = sum over the channel tiles' partials in tile order (overwrite).
// The other blocks: 32 columns of the dA / dD / d dt_bias partial rows each;
// thread (x, y) adds rows y, y+8, ... in ascending order, then the eight sums
// are added y = 0..7 (the order colsum_kernel uses).
template <int N>
__global__ void __launch_bounds__(256) ss_bwd_reduce_kernel(const float* __restrict__ ws_dBC, float* dB, float* dC,
                                                            long long nBC, int ndt, int nblk_bc,
                                                            const float* __restrict__ ws_dAD, long long nAD, int rows,
                                                            DADStore st) {
  pdl_wait();  // the partials come from the backward kernel before
  if ((int)blockIdx.x < nblk_bc) {
    for (long long i = blockIdx.x * 256ll + threadIdx.x; i < nBC; i += (long long)nblk_bc * 256) {
      float acc = 0.f;
#pragma unroll 8
      for (int t = 0; t < ndt; ++t) acc += ws_dBC[(size_t)t * nBC + i];  // loads ahead, adds in tile order
      const long long row = i / (2 * N);
      const int c = (int)(i % (2 * N));
      if (c < N) dB[row * N + c] = acc;
      else dC[row * N + (c - N)] = acc;
    }
    return;
  }
  __shared__ float red[8][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const long long i = (long long)(blockIdx.x - nblk_bc) * 32 + tx;
  float acc = 0.f;
  if (i < nAD) {
#pragma unroll 4
    for (int g = ty; g < rows; g += 8) acc += ws_dAD[(size_t)g * nAD + i];
  }
  red[ty][tx] = acc;
  __syncthreads();
  if (ty == 0 && i < nAD) {
    float v = red[0][tx];
#pragma unroll
    for (int y = 1; y < 8; ++y) v += red[y][tx];
    st.put(i, v);
  }
}

// Channels per CTA of a launch: with a recompute pass (chunk > 8) the TMEM
// columns a CTA holds grow with the chunk; from 128 columns (at most four CTAs
// per SM) a CTA takes 64 channels so that its four warps use all 128 TMEM lanes.
inline int bwd_channels(int N, int chunk) {
  const int dt = N == 4 ? bwd_dt<4>() : N == 8 ? bwd_dt<8>() : bwd_dt<16>();
  return (chunk != kS && tmem_cols(chunk) >= 128u) ? 64 : dt;
}

inline int bwd_seg_unit(int chunk) { return chunk > kTT ? chunk : kTT; }

struct BwdPlan {
  int ndt, gy, pmax;
  int ngr;  // dB/dC partial tiles: one per channel tile, or per window group of a tile
  size_t off_dAD, off_gsum, off_dsum, off_gin, total;
};

inline BwdPlan make_plan(int B, int L, int D, int N, int chunk) {
  BwdPlan pl;
  pl.ndt = (D + bwd_channels(N, chunk) - 1) / bwd_channels(N, chunk);
  pl.ngr = pl.ndt * bwd_groups(N, bwd_channels(N, chunk));
  const int cap = 1024 / pl.ndt > 0 ? 1024 / pl.ndt : 1;
  pl.gy = B < cap ? B : cap;
  const long long ctas = (long long)pl.ndt * B;
  pl.pmax = ctas >= 608 ? 1 : seg_pmax(ctas, L, bwd_seg_unit(chunk));
  const int rows = pl.pmax > 1 && B * pl.pmax > pl.gy ? B * pl.pmax : pl.gy;
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  pl.off_dAD = up((size_t)pl.ngr * B * L * 2 * N * sizeof(float));
  pl.off_gsum = up(pl.off_dAD + (size_t)rows * D * (N + 2) * sizeof(float));
  const size_t st = pl.pmax > 1 ? (size_t)B * pl.pmax * D * N * sizeof(float) : 0;
  pl.off_dsum = up(pl.off_gsum + st);
  pl.off_gin = up(pl.off_dsum + (pl.pmax > 1 ? (size_t)B * pl.pmax * D * sizeof(float) : 0));
  pl.total = pl.off_gin + st;
  return pl;
}

// pipeline depth: a staging slot is released right after the tile's widening
// pass and refilled with the next tile, which then lands during this tile's
// windows: one slot suffices (two measured no faster, and cost 5 KB a CTA)
template <typename T>
struct Stages {
  static constexpr int value = 1;
};
// the summary kernel's tiles take a few hundred cycles each: four in flight per one-warp CTA
constexpr int kSumStages = 4;

template <int N, typename T, int NSTG, int DT, bool FUSE>
int launch_bwd_f(BwdParams p, const void* x, const void* delta, const void* Bm, const void* Cm, const void* z, const void* dy,
                 float* dA, float* dB, float* dC, float* dD, void* ws, cudaStream_t stream) {
  constexpr int e = ActT<T>::kBytes;
  const BwdPlan pl = make_plan(p.B, p.L, p.D, N, p.chunk);
  p.ws_dBC = static_cast<float*>(ws);
  p.ws_dAD = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.off_dAD);
  p.gsum = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.off_gsum);
  p.dsum = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.off_dsum);
  p.gin = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.off_gin);
  p.tcols = p.chunk == kS ? 0u : tmem_cols(p.chunk);
  CUtensorMap tm[6];
  const uint64_t adims[3] = {(uint64_t)p.D, (uint64_t)p.L, (uint64_t)p.B};
  const uint64_t astr[2] = {(uint64_t)p.D * e, (uint64_t)p.L * p.D * e};
  const uint32_t abox[3] = {DT, kTT, 1};
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
  const size_t smem = sizeof(BwdSmem<T, N, NSTG, DT>);
  auto kern = scan_bwd_kernel<N, T, NSTG, DT, FUSE>;
  // TMEM: the CTAs resident on one SM must fit in its 512 columns, else an
  // allocation would wait for another CTA to finish.  Ask for enough shared
  // memory per CTA to keep the residency within that bound.
  size_t smem_launch = smem;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return SS_ERR_CUDA;
  // prefer the largest shared-memory carveout, so that residency (and the occupancy
  // query the segment and grid choices rely on) is limited by the CTAs' own needs
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  int per_sm = 0;
  per_sm = resident_ctas(kern, Geo<N, DT>::NT, smem);
  if (per_sm < 1) return SS_ERR_CUDA;
  if (p.tcols != 0 && (uint32_t)per_sm * p.tcols > 512u) {
    const int max_ctas = 512 / (int)p.tcols;
    smem_launch = (size_t)(227 * 1024) / (size_t)(max_ctas + 1) + 1024;
    if (smem_launch < smem) smem_launch = smem;
    if (smem_launch > 227 * 1024) smem_launch = 227 * 1024;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_launch) != cudaSuccess)
      return SS_ERR_CUDA;
    per_sm = resident_ctas(kern, Geo<N, DT>::NT, smem_launch);
    if (per_sm < 1) return SS_ERR_CUDA;
    if ((uint32_t)per_sm * p.tcols > 512u) return SS_ERR_UNSUPPORTED;
  }
  // segments: only when (batch row, channel tile) pairs leave resident CTA slots idle
  p.P = 1;
  p.Ls = p.L;
  if (pl.pmax > 1) {
    const long long resident = (long long)per_sm * device_sm_count();
    int want = (int)(resident / ((long long)pl.ndt * p.B));
    if (want > pl.pmax) want = pl.pmax;
    const SegPlan sp = seg_plan(want, p.L, bwd_seg_unit(p.chunk));
    p.P = sp.P;
    p.Ls = sp.Ls;
    p.sum_stride = sp.P;
  }
  // CTA rows walk their batch rows: one wave of equal CTAs when the rows do not fit at once
  // (at most pl.gy, the dA/dD partial rows the workspace holds)
  int rows = balanced_rows(p.B, pl.ndt, (long long)per_sm * device_sm_count());
  if (rows > pl.gy) rows = pl.gy;
  if (p.P > 1) {
    rows = p.B * p.P;
    constexpr int SDT = sum_dt<N>();
    const uint32_t sbox[3] = {SDT, kTT, 1};
    CUtensorMap ts[3];  // delta, z, dy in the summary's narrower boxes
    if (!ssh::encode_tiled(&ts[0], ActT<T>::kTma, 3, delta, adims, astr, sbox) ||
        !ssh::encode_tiled(&ts[1], ActT<T>::kTma, 3, z, adims, astr, sbox) ||
        !ssh::encode_tiled(&ts[2], ActT<T>::kTma, 3, dy, adims, astr, sbox))
      return SS_ERR_CUDA;
    const size_t smem_s = sizeof(BwdSumSmem<T, N, kSumStages, SDT>);
    auto skern = scan_bwd_summary_kernel<N, T, kSumStages, SDT, FUSE>;
    if (cudaFuncSetAttribute(skern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_s) != cudaSuccess)
      return SS_ERR_CUDA;
  // prefer the largest shared-memory carveout, so that residency (and the occupancy
  // query the segment and grid choices rely on) is limited by the CTAs' own needs
  cudaFuncSetAttribute(skern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    skern<<<dim3((p.D + SDT - 1) / SDT, p.B * (p.P - 1)), GeoS<N, SDT>::NT, smem_s, stream>>>(p, ts[0], ts[1], ts[2],
                                                                                           tm[5]);
    if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
    if (seg_combine<true>(SegCombine{p.A, p.dsum, p.gsum, p.dh_last, p.gin, p.P, p.D, N, p.P, 1}, p.B, stream) != cudaSuccess)
      return SS_ERR_CUDA;
  }
  kern<<<dim3(pl.ndt, rows), Geo<N, DT>::NT, smem_launch, stream>>>(p, tm[0], tm[1], tm[2], tm[3], tm[4], tm[5]);
  if (cudaGetLastError() != cudaSuccess) return SS_ERR_CUDA;
  const long long nBC = (long long)p.B * p.L * 2 * N;
  long long blk_bc = (nBC + 255) / 256;
  if (blk_bc > 8192) blk_bc = 8192;
  const long long nA = (long long)p.D * N, nAD = nA + 2ll * p.D;
  const long long blk_ad = (nAD + 31) / 32;
  const cudaError_t err = launch_dependent(ss_bwd_reduce_kernel<N>, dim3((unsigned)(blk_bc + blk_ad)), dim3(256), 0, stream,
                                         (const float*)p.ws_dBC, dB, dC, nBC, pl.ngr, (int)blk_bc, (const float*)p.ws_dAD,
                                         nAD, rows, DADStore{dA, dD, p.d_dt_bias, nA, p.D});
  return err == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// the discretisation of delta is a template switch, so the plain scan carries none of it
template <int N, typename T, int NSTG = Stages<T>::value, int DT = bwd_dt<N>()>
int launch_bwd(const BwdParams& p, const void* x, const void* delta, const void* Bm, const void* Cm, const void* z,
               const void* dy, float* dA, float* dB, float* dC, float* dD, void* ws, cudaStream_t stream) {
  return p.fuse ? launch_bwd_f<N, T, NSTG, DT, true>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, ws, stream)
                : launch_bwd_f<N, T, NSTG, DT, false>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, ws, stream);
}

int validate_bwd(int B, int L, int D, int N, int chunk, int dtype) {
  if (B <= 0 || L <= 0 || D <= 0 || N <= 0 || chunk <= 0) return SS_ERR_DIM;
  if (N != 4 && N != 8 && N != 16) return SS_ERR_UNSUPPORTED;
  if (dtype != SS_F32 && dtype != SS_BF16) return SS_ERR_UNSUPPORTED;
  if ((chunk != kS && chunk % kTT != 0) || chunk > kMaxChunk) return SS_ERR_UNSUPPORTED;
  if (D % 8 != 0) return SS_ERR_ALIGN;
  if (((long long)L * N * (dtype == SS_F32 ? 4 : 2)) % 16 != 0) return SS_ERR_ALIGN;
  if ((long long)L * N >= (1ll << 31) || (long long)L * D >= (1ll << 40)) return SS_ERR_DIM;
  return SS_OK;
}

// One whole sequence summarised: the backward summary pass over the single segment [0, L) per batch row.
template <int N, typename T, bool FUSE>
int launch_bwd_summary(BwdParams p, const void* delta, const void* Cm, const void* z, const void* dy, cudaStream_t stream) {
  constexpr int e = ActT<T>::kBytes;
  constexpr int SDT = sum_dt<N>();
  const uint64_t adims[3] = {(uint64_t)p.D, (uint64_t)p.L, (uint64_t)p.B};
  const uint64_t astr[2] = {(uint64_t)p.D * e, (uint64_t)p.L * p.D * e};
  const uint32_t sbox[3] = {SDT, kTT, 1};
  const uint64_t bdims[2] = {(uint64_t)p.L * N, (uint64_t)p.B};
  const uint64_t bstr[1] = {(uint64_t)p.L * N * e};
  const uint32_t bbox[2] = {kTT * N, 1};
  CUtensorMap tm[4];
  if (!ssh::encode_tiled(&tm[0], ActT<T>::kTma, 3, delta, adims, astr, sbox) ||
      !ssh::encode_tiled(&tm[1], ActT<T>::kTma, 3, z, adims, astr, sbox) ||
      !ssh::encode_tiled(&tm[2], ActT<T>::kTma, 3, dy, adims, astr, sbox) ||
      !ssh::encode_tiled(&tm[3], ActT<T>::kTma, 2, Cm, bdims, bstr, bbox))
    return SS_ERR_CUDA;
  const size_t smem_s = sizeof(BwdSumSmem<T, N, kSumStages, SDT>);
  auto skern = scan_bwd_summary_kernel<N, T, kSumStages, SDT, FUSE>;
  if (cudaFuncSetAttribute(skern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_s) != cudaSuccess)
    return SS_ERR_CUDA;
  cudaFuncSetAttribute(skern, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  p.P = 2;  // one summarised segment per batch row, starting at step 0
  p.Ls = p.L;
  p.sum_stride = 1;
  p.sum_first = 0;
  skern<<<dim3((p.D + SDT - 1) / SDT, p.B), GeoS<N, SDT>::NT, smem_s, stream>>>(p, tm[0], tm[1], tm[2], tm[3]);
  return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

template <int N, typename T>
int bwd_summary_fuse(const BwdParams& p, const void* delta, const void* Cm, const void* z, const void* dy, cudaStream_t s) {
  return p.fuse ? launch_bwd_summary<N, T, true>(p, delta, Cm, z, dy, s)
                : launch_bwd_summary<N, T, false>(p, delta, Cm, z, dy, s);
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
  return make_plan(B, L, D, N, chunk).total;
}

extern "C" int ss_scan_bwd(const void* x, const void* delta, const float* A, const void* Bm, const void* Cm, const float* Dv,
                           const void* z, const float* ckpt, const void* dy, const float* dh_last, float* dx, float* ddelta,
                           float* dz, float* dA, float* dB, float* dC, float* dD, float* dh0, int B, int L, int D, int N,
                           int chunk, int dtype, const float* dt_bias, int delta_softplus, float* d_dt_bias,
                           void* workspace, size_t ws_bytes, void* stream) {
  if (!x || !delta || !A || !Bm || !Cm || !Dv || !z || !ckpt || !dy || !dx || !ddelta || !dz || !dA || !dB || !dC || !dD)
    return SS_ERR_NULL;
  const int v = validate_bwd(B, L, D, N, chunk, dtype);
  if (v != SS_OK) return v;
  const void* ptrs[] = {x, delta, A, Bm, Cm, Dv, z, ckpt, dy, dx, ddelta, dz, dA, dB, dC, dD};
  for (const void* q : ptrs)
    if (!ssh::aligned16(q)) return SS_ERR_ALIGN;
  if ((dh_last && !ssh::aligned16(dh_last)) || (dh0 && !ssh::aligned16(dh0))) return SS_ERR_ALIGN;
  const BwdPlan pl = make_plan(B, L, D, N, chunk);
  if (workspace == nullptr || ws_bytes < pl.total) return SS_ERR_WORKSPACE;
  if (!ssh::aligned16(workspace)) return SS_ERR_ALIGN;
  BwdParams p{A, Dv, ckpt, dh_last, dx, ddelta, dz, dh0, nullptr, nullptr, B, L, D, chunk, ss_scan_num_chunks(L, chunk), 0,
              1, L, nullptr, nullptr, nullptr, 1, 1, dt_bias, delta_softplus ? 1 : 0,
              (dt_bias != nullptr || delta_softplus) ? 1 : 0, d_dt_bias};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool wide = bwd_channels(N, chunk) == 64;
  if (dtype == SS_F32) {
    if (N == 4) return launch_bwd<4, float>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
    if (N == 8)
      return wide ? launch_bwd<8, float, Stages<float>::value, 64>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s)
                  : launch_bwd<8, float>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
    return wide ? launch_bwd<16, float, Stages<float>::value, 64>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s)
                : launch_bwd<16, float>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
  }
  if (N == 4) return launch_bwd<4, __nv_bfloat16>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
  if (N == 8)
    return wide ? launch_bwd<8, __nv_bfloat16, Stages<__nv_bfloat16>::value, 64>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s)
                : launch_bwd<8, __nv_bfloat16>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
  return wide ? launch_bwd<16, __nv_bfloat16, Stages<__nv_bfloat16>::value, 64>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s)
              : launch_bwd<16, __nv_bfloat16>(p, x, delta, Bm, Cm, z, dy, dA, dB, dC, dD, workspace, s);
}

extern "C" int ss_scan_bwd_summary(const void* delta, const float* A, const void* Cm, const void* z, const void* dy,
                                   float* g_start, float* delta_sum, int B, int L, int D, int N, int dtype,
                                   const float* dt_bias, int delta_softplus, void* stream) {
  if (!delta || !A || !Cm || !z || !dy || !g_start || !delta_sum) return SS_ERR_NULL;
  const int v = validate_bwd(B, L, D, N, kTT, dtype);
  if (v != SS_OK) return v;
  const void* ptrs[] = {delta, A, Cm, z, dy, g_start, delta_sum};
  for (const void* q : ptrs)
    if (!ssh::aligned16(q)) return SS_ERR_ALIGN;
  BwdParams p{A, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, B, L, D, kTT, 0, 0,
              2, L, g_start, delta_sum, nullptr, 1, 0, dt_bias, delta_softplus ? 1 : 0,
              (dt_bias != nullptr || delta_softplus) ? 1 : 0, nullptr};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SS_F32) {
    if (N == 4) return bwd_summary_fuse<4, float>(p, delta, Cm, z, dy, s);
    if (N == 8) return bwd_summary_fuse<8, float>(p, delta, Cm, z, dy, s);
    return bwd_summary_fuse<16, float>(p, delta, Cm, z, dy, s);
  }
  if (N == 4) return bwd_summary_fuse<4, __nv_bfloat16>(p, delta, Cm, z, dy, s);
  if (N == 8) return bwd_summary_fuse<8, __nv_bfloat16>(p, delta, Cm, z, dy, s);
  return bwd_summary_fuse<16, __nv_bfloat16>(p, delta, Cm, z, dy, s);
}
