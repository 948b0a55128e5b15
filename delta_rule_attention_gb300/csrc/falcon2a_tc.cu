// Falcon-2A forward in chunk form on the tensor cores (bf16, m = d_v = 64,
// chunk 64).
//
// Page hyper.ai/fr/papers/2608.27763, Section 4.3 ("Falcon-2A: per-column
// inner-product write") with the per-column step sizes of Section 4.2: every
// value column j has its own step eta_{j,t} = beta_{j,t} / (||x_t||^2 +
// lambda_t + eps) and clamped decay gamma_{j,t}, and
//   s_j <- gamma_{j,t} s_j + eta_{j,t} v_{t,j} x_t,   o_{t,j} = s_j^T phi(q_t).
// There is no solve: with G_{j,t} the chunk-local log prefix of column j, a
// chunk entered with state S gives
//   o_{t,j}  = e^{G_{j,t}} (Q S)_{t,j} + sum_{s<=t} <q_t, x_s> e^{G_{j,t} - G_{j,s}} eta_{j,s} v_{s,j}
//   S'_{:,j} = e^{G_{j,C}} S_{:,j}   + sum_s x_s e^{G_{j,C} - G_{j,s}} eta_{j,s} v_{s,j}.
// The decays differ per column, so the chunk's map is elementwise in the
// state: S' = S o e^{G_C} + Nc_top and O = E o (Q S) + Nc_bot with
// E_{t,j} = e^{G_{j,t}}.
//
// tc_falcon2a_map_kernel, one CTA per (head, chunk), two per SM:
//   D1 = [Q; .] X^T (tcgen05), A = causal part of D1;
//   Nc_bot = F o (A U~), U~_{s,j} = e^{r_j - G_{j,s}} eta_{j,s} v_{s,j},
//            F_{t,j} = e^{G_{j,t} - r_j}, r_j = G_{j,C} / 2 (both factors stay
//            within fp32 range while -G_{j,C} <= 160; a chunk with a longer
//            decay span forms Nc_bot directly on the CUDA cores instead);
//   Nc_top = X^T V', V'_{s,j} = e^{G_{j,C} - G_{j,s}} eta_{j,s} v_{s,j}.
//   The map (phi(Q), Nc, E as bf16 operand images, e^{G_C} in fp32) goes to
//   the workspace.
// tc_falcon2a_scan_kernel, one CTA per head, sequential over chunks: the
//   state update is elementwise (fp32 registers); per chunk one tcgen05 MMA
//   forms Q S for the output rows.
#include <cuda_bf16.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"
#include "tmap.cuh"

namespace falcon {

namespace {

using namespace tc;
using namespace tcu;

constexpr int k2C = 64;
constexpr int k2Threads = 256;
constexpr uint32_t k2Tile = 8192;
// Map of one (head, chunk): phi(Q) | Nc (state rows, then output rows) | E | e^{G_C}.
constexpr uint32_t kM2Q = 0, kM2Nc = 8192, kM2E = 24576, kM2G = 32768;
constexpr uint32_t kMap2ABytes = kM2G + 256;
constexpr float kSpan2A = 160.f;

// Map kernel tiles: X, Q, V, A (causal Q X^T), U~, V'.  The map stages reuse
// the dead ones: Nc over A and U~, E over V'.
enum : int { kX2 = 0, kQ2, kV2, kA2, kU2, kVp2, k2Slots };
constexpr int kLdG = 65;
constexpr uint32_t kBetaOff = k2Slots * k2Tile;      // beta rows as copied (fp32, 64 x 64)
constexpr uint32_t kEtaOff = kBetaOff + 64 * 64 * 4;  // eta (fp32, 64 x kLdG)
constexpr uint32_t kGOff = kEtaOff + 64 * kLdG * 4;   // G (fp32, 64 x kLdG)
constexpr uint32_t kSc2Off = kGOff + 64 * kLdG * 4;

struct F2Scalars {
  float E[64], inv[64], lam[64], r[64], gC[64], half[64];  // inv: 1 / (E + lambda + eps), 0 if none
  float part[4][64];  // column sums of the four quarters of the token range
  float ssp[2][128];
  int fail, slow;
  uint64_t bar_in, bar_mma;
  uint32_t tmem_base;
};
constexpr size_t kF2Smem = kSc2Off + sizeof(F2Scalars) + 1024;
static_assert(2 * (kF2Smem + 1024) <= 228 * 1024, "two CTAs per SM");

__device__ __forceinline__ void publish_f2() {
  tc_fence_before();
  fence_async_smem();
  __syncthreads();
}

__global__ void __launch_bounds__(k2Threads, 2)
    tc_falcon2a_map_kernel(ChunkArgs a, int nchunks, int* err,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = align1024(smem_raw);
  float* Beta = reinterpret_cast<float*>(base + kBetaOff);  // [t][j], as copied
  float* Eta = reinterpret_cast<float*>(base + kEtaOff);    // [t][j], rows of kLdG
  float* G = reinterpret_cast<float*>(base + kGOff);        // log gamma, then the prefix
  F2Scalars& sc = *reinterpret_cast<F2Scalars*>(base + kSc2Off);
  auto tile = [&](int i) { return base + i * k2Tile; };
  auto taddr = [&](int i) { return smem_addr(base + i * k2Tile); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, h = tid >> 7;
  const int c = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t T = a.T, t0 = (int64_t)c * k2C, rowbase = bh * T;
  const int n = (int)min((int64_t)k2C, T - t0);

  // TMEM is allocated by warp 1, so that thread 0 issues the input tile copies
  // (the head of the CTA's chain) without waiting for the allocation.
  if (warp == 1) tmem_alloc(&sc.tmem_base, 256);
  // Launched behind the previous call's scan (programmatic dependent launch):
  // nothing is read or written before the preceding grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    mbar_init(&sc.bar_in, 1);
    mbar_init(&sc.bar_mma, 1);
    fence_mbar_init();
    sc.fail = 0;
    sc.slow = 0;
    // k rows t0-1 .. t0+62, q and v rows t0 .. (zeros outside), beta rows t0 ..
    mbar_expect_tx(&sc.bar_in, 3 * k2Tile + (uint32_t)n * 256u);
    tma_load_3d(tile(kX2), &tm_k, 0, (int)(t0 - 1), (int)bh, &sc.bar_in);
    tma_load_3d(tile(kQ2), &tm_q, 0, (int)t0, (int)bh, &sc.bar_in);
    tma_load_3d(tile(kV2), &tm_v, 0, (int)t0, (int)bh, &sc.bar_in);
    bulk_g2s(Beta, a.beta + (rowbase + t0) * 64, (uint32_t)n * 256u, &sc.bar_in);
  }
  if (tid < 64) sc.lam[tid] = tid < n ? a.lambda[rowbase + t0 + tid] : 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sc.tmem_base;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * h;
  uint32_t phase = 0;
  bool slow = false;
  if (!mbar_wait_backoff(&sc.bar_in, 0)) sc.fail = 1;
  if (__syncthreads_or(sc.fail)) goto teardown;

  // ---- features: rows 0..63 of [X; Q] are x_t = phi(k_{t-1}) (x_prev, or the
  //      sentinel zero, at t = 0), rows 64..127 are phi(q_t); rows past the
  //      chunk's tokens are zero.
  {
    float v[32];
    load_half_sw(tile(kX2), r, h, v);
    const int i = r & 63;
    const bool xrow = r < 64;
    const bool given = xrow && t0 + i == 0 && a.x_prev != nullptr;
    const bool dead = i >= n || (xrow && t0 + i == 0 && a.x_prev == nullptr);
    if (given)
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = a.x_prev[bh * 64 + 32 * h + j];
    sc.ssp[h][r] = sumsq32(v);
    __syncthreads();
    const float ss = sc.ssp[0][r] + sc.ssp[1][r];
    const float s = dead ? 0.f : (given ? 1.f : phi_scale(ss, 64, a.phi));
    store_half_sw(tile(kX2), r, h, v, s);
    if (xrow && h == 0) sc.E[i] = ss * s * s;
  }
  __syncthreads();
  if (tid < 64) {
    // The step-size denominator is shared by the token's columns: one
    // reciprocal per token (0 for the sentinel and a non-positive denominator).
    const float lam = ridge_of(sc.lam[tid], sc.E[tid], a.ridge);
    sc.lam[tid] = lam;
    const float den = sc.E[tid] + lam + a.eps;
    const bool sentinel = (t0 + tid == 0) && (a.x_prev == nullptr);
    sc.inv[tid] = (!sentinel && den > 0.f) ? 1.f / den : 0.f;
  }
  __syncthreads();
  // ---- eta_{j,t} and log gamma_{j,t} per (token, column) (the decay clamp of
  //      step_eta_gamma: gamma = eps_gamma exactly on the clamped branch), then
  //      the prefix down each column
  {
    const float lg_clamped = logf(a.eps_gamma);
    for (int idx = tid; idx < 64 * 64; idx += k2Threads) {
      const int t = idx >> 6, j = idx & 63;
      float eta = 0.f, lg = 0.f;
      if (t < n) {
        eta = Beta[idx] * sc.inv[t];
        const float al = eta * sc.lam[t];
        lg = al >= 1.f - a.eps_gamma ? lg_clamped : log1pf(-al);
      }
      Eta[t * kLdG + j] = eta;
      G[t * kLdG + j] = lg;
    }
  }
  __syncthreads();
  {
    // column prefixes: thread (j, p) sums tokens 16p .. 16p + 15 of column j,
    // then adds the sums of the quarters before it
    const int j = tid & 63, p = tid >> 6;
    float run = 0.f;
#pragma unroll
    for (int t = 16 * p; t < 16 * p + 16; ++t) {
      run += G[t * kLdG + j];
      G[t * kLdG + j] = run;
    }
    sc.part[p][j] = run;
    __syncthreads();
    float off = 0.f;
    for (int q = 0; q < p; ++q) off += sc.part[q][j];
    if (p > 0)
#pragma unroll
      for (int t = 16 * p; t < 16 * p + 16; ++t) G[t * kLdG + j] += off;
    if (p == 3) {
      const float gc = off + run;
      sc.gC[j] = gc;
      sc.r[j] = 0.5f * gc;
      sc.half[j] = __expf(0.5f * gc);  // e^{G_C - r}
      if (-gc > kSpan2A) atomicOr(&sc.slow, 1);
    }
  }
  publish_f2();
  slow = sc.slow != 0;

  // ---- D1 = [Q; .] X^T (rows 64..127 of the A operand read the V tile)
  if (tid == 0) {
    tc_fence_after();
    mma_k64(tmem, taddr(kQ2), false, 16, taddr(kX2), false, 16,
            idesc_bf16(128, 64, false, false), false);
    mma_commit(&sc.bar_mma);
  }
  // U~ and V' rows (thread: row s = r & 63, column half h; r < 64: U~, else V')
  {
    const int s = r & 63;
    float v[32];
    load_half_sw(tile(kV2), s, h, v);
    float u[32];
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const int j = 32 * h + jj;
      const float ev = Eta[s * kLdG + j] * v[jj];
      if (slow) {
        u[jj] = 0.f;
        v[jj] = __expf(fminf(sc.gC[j] - G[s * kLdG + j], 0.f)) * ev;
      } else {
        // U~ = e^{r - G_s} eta v; V' = e^{G_C - G_s} eta v = e^{G_C - r} U~
        u[jj] = __expf(sc.r[j] - G[s * kLdG + j]) * ev;
        v[jj] = sc.half[j] * u[jj];
      }
    }
    store_half_sw(tile(r < 64 ? kU2 : kVp2), s, h, r < 64 ? u : v, 1.f);
  }
  if (!mbar_wait_backoff(&sc.bar_mma, phase)) sc.fail = 1;
  phase ^= 1u;
  tc_fence_after();
  // No barrier: each thread has seen the MMA complete before it reads its
  // accumulator rows; a failed wait is agreed on at the next barrier.
  // A = causal part of Q X^T (rows 0..63: lanes of warps 0, 1, 4, 5)
  if ((warp & 3) < 2) {
    float d[32];
    tmem_ld32(tl, d);
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) d[jj] = (32 * h + jj <= r) ? d[jj] : 0.f;
    store_half_sw(tile(kA2), r, h, d, 1.f);
  }
  tc_fence_before();
  fence_async_smem();
  if (__syncthreads_or(sc.fail)) goto teardown;
  // ---- D2 = A U~ (output rows), D3 = X^T V' (state rows)
  if (tid == 0) {
    tc_fence_after();
    mma_k64(tmem + 64, taddr(kA2), false, 16, taddr(kU2), true, k2Tile,
            idesc_bf16(128, 64, false, true), false);
    mma_k64(tmem + 128, taddr(kX2), true, k2Tile, taddr(kVp2), true, k2Tile,
            idesc_bf16(128, 64, true, true), false);
    mma_commit(&sc.bar_mma);
  }
  if (!mbar_wait_backoff(&sc.bar_mma, phase)) sc.fail = 1;
  phase ^= 1u;
  tc_fence_after();
  // No barrier: each thread has seen the MMAs complete before it overwrites
  // their operands with the staging; a failed wait is agreed on below.
  // ---- the map: phi(Q) (the Q tile itself), Nc (state rows from D3, output
  //      rows F o D2) over the A and U~ tiles, E over the V' tile, e^{G_C}
  {
    unsigned char* nc_stage = tile(kA2);  // 16 KB: kA2, kU2
    unsigned char* e_stage = tile(kVp2);
    if ((warp & 3) < 2) {
      const int t = r;
      float d[32], o[32];
      tmem_ld32(tl + 128, d);
      tmem_ld32(tl + 64, o);
      if (slow) {
        // sum_{s<=t} <q_t, x_s> e^{G_{j,t} - G_{j,s}} eta_{j,s} v_{s,j}, directly
        float qx[64];
        tmem_ld32(tl - 32 * h, qx);
        tmem_ld32(tl - 32 * h + 32, qx + 32);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) o[jj] = 0.f;
        for (int s = 0; s <= t; ++s) {
          float v[32];
          load_half_sw(tile(kV2), s, h, v);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int j = 32 * h + jj;
            o[jj] += qx[s] * __expf(fminf(G[t * kLdG + j] - G[s * kLdG + j], 0.f)) *
                     Eta[s * kLdG + j] * v[jj];
          }
        }
      }
      // (rows past the chunk's tokens: q_t = 0, so their o rows are zero)
      float e[32];
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) e[jj] = __expf(G[t * kLdG + 32 * h + jj]);
      if (!slow) {
        // F = e^{G_t - r}: E / e^{r} would overflow nothing but lose range when
        // e^{G_t} underflows, so it takes its own exponential
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = 32 * h + jj;
          o[jj] *= __expf(G[t * kLdG + j] - sc.r[j]);
        }
      }
      __syncwarp();
      // Writing over A and U~ is safe: both MMAs that read them have completed.
      store_half_sw(nc_stage, t, h, d, 1.f);
      store_half_sw(nc_stage, 64 + t, h, o, 1.f);
      store_half_sw(e_stage, t, h, e, 1.f);
    }
    fence_async_smem();
    if (__syncthreads_or(sc.fail)) goto teardown;
    if (tid == 0) {
      unsigned char* map = reinterpret_cast<unsigned char*>(a.workspace) +
                           (size_t)(bh * nchunks + c) * kMap2ABytes;
      bulk_s2g(map + kM2Q, tile(kQ2), k2Tile);
      bulk_s2g(map + kM2Nc, nc_stage, 2 * k2Tile);
      bulk_s2g(map + kM2E, e_stage, k2Tile);
      bulk_commit();
    }
    if (tid >= 64 && tid < 128) {
      float* gdst = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(a.workspace) +
                                             (size_t)(bh * nchunks + c) * kMap2ABytes + kM2G);
      gdst[tid - 64] = __expf(sc.gC[tid - 64]);
    }
    if (tid == 0) bulk_wait_read<0>();
    // x_last = phi(k_{T-1}) (last chunk, one warp)
    if (a.x_last && c == nchunks - 1 && warp == 7) {
      const __nv_bfloat16* kl = reinterpret_cast<const __nv_bfloat16*>(a.k) + (rowbase + T - 1) * 64;
      const float u0 = __bfloat162float(kl[lane]), u1 = __bfloat162float(kl[lane + 32]);
      const float s = phi_scale(warp_sum(u0 * u0 + u1 * u1), 64, a.phi);
      a.x_last[bh * 64 + lane] = u0 * s;
      a.x_last[bh * 64 + lane + 32] = u1 * s;
    }
  }

teardown:
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (sc.fail && tid == 0) atomicExch(err, 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// Scan: one CTA per head.  Threads of warps 0, 1, 4, 5 own state row
// k = 32 (w & 3) + lane, columns 32 (w >> 2) .. +31 (fp32 registers), and the
// same output row t = k of every chunk; lane 0 of warp 2 loads the maps (a
// ring of kS2Stages) and issues the MMAs.  Per chunk: the state goes to the
// operand tile as bf16, the MMA [Q; .] S starts, the state update
// S <- S o e^{G_C} + Nc_top runs meanwhile, then o = E o (Q S) + Nc_bot leaves
// by a TMA store.
constexpr int kS2Stages = 4;
constexpr uint32_t kS2Stage = 4 * k2Tile;  // phi(Q) | Nc (two tiles) | E

struct S2Smem {
  unsigned char stage[kS2Stages][kS2Stage];
  unsigned char sop[k2Tile];     // S (bf16) as the MN-major B operand
  unsigned char ost[2][k2Tile];  // o tiles for the TMA store
  float gc[kS2Stages][64];
  uint64_t full[kS2Stages];
  uint64_t bar_mma;
  uint32_t tmem_base;
  int fail;
};

__device__ __forceinline__ void s2_issue_load(S2Smem& s, int st, const unsigned char* map) {
  mbar_expect_tx(&s.full[st], kS2Stage + 256);
  bulk_g2s(s.stage[st], map, kS2Stage, &s.full[st]);
  bulk_g2s(s.gc[st], map + kM2G, 256, &s.full[st]);
}

// Half row h (32 values) of row `row` of a swizzled stage tile.
__device__ __forceinline__ void ld_row32(const unsigned char* tile, int row, int h, float* v) {
  load_half_sw(tile, row, h, v);
}

__global__ void __launch_bounds__(k2Threads, 1)
    tc_falcon2a_scan_kernel(ChunkArgs a, int nchunks, int* err,
                            const __grid_constant__ CUtensorMap tm_o) {
  extern __shared__ unsigned char smem_raw[];
  S2Smem& s = *reinterpret_cast<S2Smem*>(align1024(smem_raw));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bh = blockIdx.x;
  const bool state = (warp & 3) < 2;
  const bool issuer = warp == 2 && lane == 0;
  const int row = 32 * (warp & 3) + lane, h = warp >> 2;
  const unsigned char* hmaps = reinterpret_cast<const unsigned char*>(a.workspace) +
                               (size_t)bh * nchunks * kMap2ABytes;
  // A following map launch may start now; it waits for this grid to complete
  // before it touches memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 0) tmem_alloc(&s.tmem_base, 64);
  if (tid == 0) {
    for (int st = 0; st < kS2Stages; ++st) mbar_init(&s.full[st], 1);
    mbar_init(&s.bar_mma, 1);
    fence_mbar_init();
    s.fail = 0;
  }
  float S[32];
  if (state) {
#pragma unroll
    for (int j = 0; j < 32; ++j) S[j] = a.S0 ? a.S0[(bh * 64 + row) * 64 + 32 * h + j] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the maps of the preceding launch
  const uint32_t tmem = s.tmem_base;
  if (issuer)
    for (int k = 0; k < kS2Stages && k < nchunks; ++k)
      s2_issue_load(s, k, hmaps + (size_t)k * kMap2ABytes);
  const uint32_t idesc = idesc_bf16(128, 64, false, true);
  for (int c = 0; c < nchunks; ++c) {
    const int st = c % kS2Stages, b = c & 1;
    unsigned char* stg = s.stage[st];
    if (state) {
      store_half_sw(s.sop, row, h, S, 1.f);
      fence_async_smem();
    }
    if (issuer && !mbar_wait(&s.full[st], (uint32_t)(c / kS2Stages) & 1u)) s.fail = 1;
    if (issuer) bulk_wait_read<1>();  // o tile b: its store of chunk c - 2 has read it
    if (__syncthreads_or(s.fail)) break;
    if (issuer) {
      tc_fence_after();
      // rows 64..127 of the A operand read the stage's Nc (lanes nobody reads)
      mma_k64(tmem, smem_addr(stg), false, 16, smem_addr(s.sop), true, k2Tile, idesc, false);
      mma_commit(&s.bar_mma);
    }
    float nco[32];
    if (state) {
      // S <- S o e^{G_C} + Nc_top (off the MMA)
      float nct[32];
      ld_row32(stg + k2Tile, row, h, nct);
      ld_row32(stg + k2Tile, 64 + row, h, nco);
#pragma unroll
      for (int j = 0; j < 32; ++j) S[j] = s.gc[st][32 * h + j] * S[j] + nct[j];
    }
    if (!mbar_wait(&s.bar_mma, (uint32_t)c & 1u)) s.fail = 1;
    tc_fence_after();
    if (__syncthreads_or(s.fail)) break;
    if (state) {
      float d[32], e[32];
      tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * h, d);
      ld_row32(stg + 3 * k2Tile, row, h, e);
#pragma unroll
      for (int j = 0; j < 32; ++j) d[j] = e[j] * d[j] + nco[j];
      store_half_sw(s.ost[b], row, h, d, 1.f);
      fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();  // o tile complete; stage st fully read
    if (issuer) {
      tma_store_3d(&tm_o, s.ost[b], 0, c * k2C, (int)bh);
      bulk_commit();
      if (c + kS2Stages < nchunks)
        s2_issue_load(s, st, hmaps + (size_t)(c + kS2Stages) * kMap2ABytes);
    }
  }
  if (issuer) bulk_wait<0>();
  if (!s.fail && state) {
    float* dst = a.S_out + (bh * 64 + row) * 64 + 32 * h;
#pragma unroll
    for (int j = 0; j < 32; ++j) dst[j] = S[j];
  }
  if (s.fail && tid == 0) atomicExch(err, 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

}  // namespace

bool tc_falcon2a_applies(int dtype, int m, int dv, int C, int64_t BH, int64_t T) {
  return tc_path_applies(dtype, m, dv, C, BH, T) && m == 64;
}

size_t tc_falcon2a_workspace_bytes(int64_t BH, int64_t T) {
  return (size_t)(BH * ((T + k2C - 1) / k2C)) * kMap2ABytes;
}

cudaError_t launch_tc_falcon2a(const ChunkArgs& a, int* err, cudaStream_t stream) {
  const int nchunks = (int)((a.T + k2C - 1) / k2C);
  CUtensorMap tm_k, tm_q, tm_v, tm_o;
  if (!encode_rows_bf16(&tm_k, a.k, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, k2C) ||
      !encode_rows_bf16(&tm_q, a.q, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, k2C) ||
      !encode_rows_bf16(&tm_v, a.v, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, k2C) ||
      !encode_rows_bf16(&tm_o, a.o, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, k2C))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_falcon2a_map_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kF2Smem);
  if (e != cudaSuccess) return e;
  // Both launches are programmatic dependent launches: the maps behind the
  // preceding kernel, the scan behind the maps; each waits (griddepcontrol.wait)
  // for its predecessor before touching memory.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(nchunks, (unsigned)a.BH);
  mcfg.blockDim = dim3(k2Threads);
  mcfg.dynamicSmemBytes = kF2Smem;
  mcfg.stream = stream;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&mcfg, tc_falcon2a_map_kernel, a, nchunks, err, tm_k, tm_q, tm_v)) !=
      cudaSuccess)
    return e;
  const size_t smem = sizeof(S2Smem) + 1024;
  e = cudaFuncSetAttribute(tc_falcon2a_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.BH);
  cfg.blockDim = dim3(k2Threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_falcon2a_scan_kernel, a, nchunks, err, tm_o);
}

}  // namespace falcon
