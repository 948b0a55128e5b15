// Falcon-3A forward in chunk form on the tensor cores (bf16, m = d_v = 64,
// chunk 64, window B <= 32), for fresh sequences.
//
// Page hyper.ai/fr/papers/2608.27763, Section 4.5 (the sliding-window rule)
// and Section 4.6 (its masked-attention form with chunk-local log decays and
// the tail of the previous B - 1 pairs).  With the write pairs (x_j, v_j),
// x_j = phi(k_{j-1}), the window I_s = {max(2, s-B+1) .. s} of token s, and
// c_s = eta_s / B_s, the state after token t unrolls to
//
//   S_t = e^{g_t} S + sum_j x_j v_j^T w_{t,j},
//   w_{t,j} = sum_{s in chunk, s <= t, j in I_s} e^{g_t - g_s} c_s,
//
// inside a chunk entered with state S (g the chunk-local log prefix).  The
// coefficients follow the recurrence w_{t,j} = gamma_t w_{t-1,j} +
// [j in I_t] c_t down each column j (no exponential of a positive
// argument), over the chunk's own pairs and the B - 1 pairs before it.  So a
// chunk is the affine map the tensor-core scan applies,
//
//   [S'; O] = Mc S + Nc,  Mc = [0; Diag(e^g) Q] (plus e^{g_C} S on the state
//   rows), Nc = [X~^T Diag(w_C) V~; (Q X~^T o W) V~],
//
// with X~, V~ the 128 pairs j = t0-64 .. t0+63 (the tail and the chunk's own;
// pairs outside every window get w = 0).  This kernel writes the map in the
// format of the Falcon-1 tensor-core forward (Mc, Nc as bf16 operand images,
// e^{g_C}); tc_chunk_scan_kernel then produces o and S_T.
//
// One CTA per (head, chunk), 256 threads, three CTAs per SM (74 KB of shared
// memory, 128 TMEM columns).  MMAs (bf16 operands in 128B-swizzled tiles,
// fp32 accumulators in TMEM):
//   D1 = [Q; .] X~^T            (N = 128: the Gram rows of the chunk's q)
//   D2 = (Q X~^T o W) V~        (K = 128 in two steps of 64)
//   D3 = X~^T Diag(w_C) V~      (X~ read MN-major, K = 128)
// D2 and D3 take the TMEM columns of D1 once it is read.
#include <cuda_bf16.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"
#include "tmap.cuh"

namespace falcon {

namespace {

using namespace tc;
using namespace tcu;

constexpr int k3C = 64;
constexpr int k3Threads = 256;
constexpr uint32_t k3Tile = 8192;
// Tile slots: X~ (two tiles: pairs t0-64 .. t0-1, t0 .. t0+63), Q, V~ (two),
// then a 32 KB region R whose contents follow each other as they die: the
// row norms' partial sums and ||x_j||^2 (features), the fp32 coefficient
// matrix W (64 x 128), then the W-masked Gram rows P (two column halves) and
// Vs = Diag(w_C) V~ (two), and last the map stages, Mc over P and Nc over Vs.
enum : int { kX0 = 0, kX1, kQ3, kV0, kV1, kP0, kP1, kVs0, kVs1, k3Slots };
constexpr uint32_t kROff = kP0 * k3Tile;  // R: the last four slots
constexpr uint32_t kSc3Off = k3Slots * k3Tile;
// W[i][j] at float i * 128 + (j ^ (i & 31)): the recurrence writes a row with
// consecutive lanes on consecutive columns and the P rows read a column run
// with consecutive lanes on consecutive rows, both without bank conflicts.
__device__ __forceinline__ int w_at(int i, int j) { return i * 128 + (j ^ (i & 31)); }

// Scalars kept beside the tiles (the features' partial sums and ||x_j||^2
// live in R while it is free).
struct F3Scalars {
  float wC[128];    // w_{C,j}: the coefficients of the state leaving the chunk
  float coef[64];   // eta_t / B_t
  float gam[64];
  float g[64], gx[64];
  int fail;
  uint64_t bar_in, bar_mma;
  uint32_t tmem_base;
};
struct F3Early {    // in R, before W
  float ssp[2][128];
  float E[128];     // ||x_j||^2 of the 128 pairs
};
static_assert(sizeof(F3Early) <= 4 * k3Tile, "features' scratch within R");
constexpr size_t kF3Smem = kSc3Off + sizeof(F3Scalars) + 1024;
static_assert(3 * (kF3Smem + 1024) <= 228 * 1024, "three CTAs per SM");

// Generic-proxy tile writes of this CTA become visible to the next MMA.
__device__ __forceinline__ void publish_tiles_f3() {
  tc_fence_before();
  fence_async_smem();
  __syncthreads();
}

__global__ void __launch_bounds__(k3Threads, 3)
    tc_falcon3a_map_kernel(ChunkArgs a, int window, int nchunks, int* err,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = align1024(smem_raw);
  float* W = reinterpret_cast<float*>(base + kROff);
  F3Scalars& sc = *reinterpret_cast<F3Scalars*>(base + kSc3Off);
  F3Early& ea = *reinterpret_cast<F3Early*>(base + kROff);
  auto tile = [&](int i) { return base + i * k3Tile; };
  auto taddr = [&](int i) { return smem_addr(base + i * k3Tile); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, h = tid >> 7;
  const int c = blockIdx.x;
  const int64_t bh = blockIdx.y;
  const int64_t T = a.T, t0 = (int64_t)c * k3C, rowbase = bh * T;
  const int n = (int)min((int64_t)k3C, T - t0);

  // TMEM is allocated by warp 1, so that thread 0 issues the input tile copies
  // (the head of the CTA's chain) without waiting for the allocation.
  if (warp == 1) tmem_alloc(&sc.tmem_base, 128);
  // Launched behind the previous call's scan (programmatic dependent launch):
  // nothing is read or written before the preceding grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    mbar_init(&sc.bar_in, 1);
    mbar_init(&sc.bar_mma, 1);
    fence_mbar_init();
    sc.fail = 0;
    // k rows t0-65 .. t0+62 (x~ of pairs t0-64 .. t0+63), q rows t0 ..,
    // v rows t0-64 .. t0+63; rows outside the sequence read zeros.
    mbar_expect_tx(&sc.bar_in, 5 * k3Tile);
    tma_load_3d(tile(kX0), &tm_k, 0, (int)(t0 - 65), (int)bh, &sc.bar_in);
    tma_load_3d(tile(kX1), &tm_k, 0, (int)(t0 - 1), (int)bh, &sc.bar_in);
    tma_load_3d(tile(kQ3), &tm_q, 0, (int)t0, (int)bh, &sc.bar_in);
    tma_load_3d(tile(kV0), &tm_v, 0, (int)(t0 - 64), (int)bh, &sc.bar_in);
    tma_load_3d(tile(kV1), &tm_v, 0, (int)t0, (int)bh, &sc.bar_in);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sc.tmem_base;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * h;
  uint32_t phase = 0;
  float gC = 0.f;
  if (!mbar_wait_backoff(&sc.bar_in, 0)) sc.fail = 1;
  if (__syncthreads_or(sc.fail)) goto teardown;

  // ---- features: row r of X~ is x_j, j = t0 - 64 + r (x_0 = 0: the boundary
  //      pair never enters a window); rows 0..63 of Q are phi(q_t).
  {
    float v[32];
    load_half_sw(tile(kX0), r, h, v);
    ea.ssp[h][r] = sumsq32(v);
    __syncthreads();
    const float ss = ea.ssp[0][r] + ea.ssp[1][r];
    const float s = phi_scale(ss, 64, a.phi);
    store_half_sw(tile(kX0), r, h, v, s);
    if (h == 0) ea.E[r] = ss * s * s;
    __syncthreads();
    const int qr = tid & 63, qh = (tid >> 6) & 1;
    if (tid < 128) {
      load_half_sw(tile(kQ3), qr, qh, v);
      ea.ssp[qh][qr] = sumsq32(v);
    }
    __syncthreads();
    if (tid < 128) {
      const float sq = ea.ssp[0][qr] + ea.ssp[1][qr];
      store_half_sw(tile(kQ3), qr, qh, v, phi_scale(sq, 64, a.phi));
    }
  }
  // ---- per token: window energy, eta_t / B_t, gamma_t (token 0 and padding:
  //      no update), then the chunk-local log prefixes
  if (tid < 64) {
    const int64_t t = t0 + tid;
    float cf = 0.f, gm = 1.f, lg = 0.f;
    if (t >= 1 && t < T) {
      const int64_t j0 = max(t - window + 1, (int64_t)1);
      const int Bt = (int)(t - j0 + 1);
      float e = 0.f;
      for (int u = 0; u < Bt; ++u) e += ea.E[64 + tid - u];
      const float Ebar = e / (float)Bt;
      const float lam = ridge_of(a.lambda[rowbase + t], Ebar, a.ridge);
      const float eta = step_eta_gamma(false, Ebar, a.beta[rowbase + t], lam, a.eps,
                                       a.eps_gamma, &gm, &lg);
      cf = eta / (float)Bt;
    }
    sc.coef[tid] = cf;
    sc.gam[tid] = gm;
    sc.g[tid] = lg;
  }
  __syncthreads();
  if (warp == 0) {
    // inclusive and exclusive prefix of the log-decays, two tokens per lane
    const float a0 = sc.g[2 * lane], a1 = sc.g[2 * lane + 1];
    float s2 = a0 + a1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, s2, o);
      if (lane >= o) s2 += y;
    }
    const float e0 = s2 - (a0 + a1);
    sc.gx[2 * lane] = e0;
    sc.gx[2 * lane + 1] = e0 + a0;
    sc.g[2 * lane] = e0 + a0;
    sc.g[2 * lane + 1] = e0 + a0 + a1;
  }
  publish_tiles_f3();
  gC = sc.g[63];

  // ---- D1 = [Q; .] X~^T (rows 64..127 of the A operand read the V0 tile)
  if (tid == 0) {
    tc_fence_after();
    mma_k64(tmem, taddr(kQ3), false, 16, taddr(kX0), false, 16,
            idesc_bf16(128, 128, false, false), false);
    mma_commit(&sc.bar_mma);
  }
  // ---- W: column j of pair j = t0 - 64 + j, w_t = gamma_t w_{t-1} + [j in I_t] c_t.
  //      Two threads per column, one per half of the chunk's tokens; the second
  //      half starts from zero and then adds (prod_{r=32}^{t} gamma_r) w_31.
  {
    const int col = tid & 127, hf = tid >> 7;
    const int64_t jg = t0 - 64 + col;
    float w = 0.f;
    for (int ii = 0; ii < 32; ++ii) {
      const int i = 32 * hf + ii;
      const int64_t t = t0 + i;
      const bool in = jg >= 1 && jg <= t && t <= jg + window - 1;
      w = sc.gam[i] * w + (in ? sc.coef[i] : 0.f);
      W[w_at(i, col)] = w;
    }
    __syncthreads();
    if (hf == 1) {
      const float w31 = W[w_at(31, col)];
      float p = 1.f;
      for (int i = 32; i < 64; ++i) {
        p *= sc.gam[i];
        W[w_at(i, col)] += p * w31;
      }
      sc.wC[col] = W[w_at(63, col)];
    }
  }
  __syncthreads();
  if (!mbar_wait_backoff(&sc.bar_mma, phase)) sc.fail = 1;
  phase ^= 1u;
  tc_fence_after();
  // P = (Q X~^T) o W, rows 0..63 (lanes 0..63), two column halves per tile:
  // every thread reads its part of W before any P row is written over W.
  {
    uint32_t pk[2][16];
    if ((warp & 3) < 2) {
      const int i = r;
      float d[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        tmem_ld32(tl + 64 * half, d);
#pragma unroll
        for (int jj = 0; jj < 32; jj += 2) {
          pk[half][jj / 2] = pack_bf16(d[jj] * W[w_at(i, 64 * half + 32 * h + jj)],
                                       d[jj + 1] * W[w_at(i, 64 * half + 32 * h + jj + 1)]);
        }
      }
    }
    tc_fence_before();
    if (__syncthreads_or(sc.fail)) goto teardown;  // W read; D1 read
    if ((warp & 3) < 2) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        unsigned char* row = tile(half ? kP1 : kP0) + r * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(row + (((4 * h + q) ^ (r & 7)) << 4)) =
              make_uint4(pk[half][4 * q], pk[half][4 * q + 1], pk[half][4 * q + 2],
                         pk[half][4 * q + 3]);
      }
    }
  }
  // Vs = Diag(w_C) V~ (rows r of the two V tiles), over the rest of W
  {
    float v[32];
    load_half_sw(tile(kV0), r, h, v);
    store_half_sw(tile(kVs0), r, h, v, sc.wC[r]);
  }
  tc_fence_before();
  fence_async_smem();
  if (__syncthreads_or(sc.fail)) goto teardown;
  // ---- D2 = P V~ (K = 128), D3 = X~^T Vs (K = 128, X~ read MN-major), in the
  //      columns D1 held
  if (tid == 0) {
    tc_fence_after();
    const uint32_t id_pv = idesc_bf16(128, 64, false, true);
    mma_k64(tmem, taddr(kP0), false, 16, taddr(kV0), true, k3Tile, id_pv, false);
    mma_k64(tmem, taddr(kP1), false, 16, taddr(kV1), true, k3Tile, id_pv, true);
    const uint32_t id_xv = idesc_bf16(128, 64, true, true);
    mma_k64(tmem + 64, taddr(kX0), true, k3Tile, taddr(kVs0), true, k3Tile, id_xv, false);
    mma_k64(tmem + 64, taddr(kX1), true, k3Tile, taddr(kVs1), true, k3Tile, id_xv, true);
    mma_commit(&sc.bar_mma);
  }
  if (!mbar_wait_backoff(&sc.bar_mma, phase)) sc.fail = 1;
  phase ^= 1u;
  tc_fence_after();
  // No barrier: each thread has seen the MMAs complete before it overwrites
  // their operands with the staging; a failed wait is agreed on below.
  // ---- the map: Mc = [0; Diag(e^g) phi(Q)] over the P tiles, Nc = [D3; D2]
  //      over the Vs tiles, e^{g_C}
  {
    unsigned char* mc_stage = tile(kP0);
    unsigned char* nc_stage = tile(kVs0);
    float v[32];
    if (r < 64) {
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) v[jj] = 0.f;
      store_half_sw(mc_stage, r, h, v, 1.f);
    } else {
      load_half_sw(tile(kQ3), r - 64, h, v);
      store_half_sw(mc_stage, r, h, v, __expf(sc.g[r - 64]));
    }
    if ((warp & 3) < 2) {
      tmem_ld32(tl + 64, v);
      store_half_sw(nc_stage, r, h, v, 1.f);
      tmem_ld32(tl, v);
      store_half_sw(nc_stage, 64 + r, h, v, 1.f);
    }
    fence_async_smem();
    if (__syncthreads_or(sc.fail)) goto teardown;
    if (tid == 0) {
      unsigned char* map = reinterpret_cast<unsigned char*>(a.workspace) +
                           (size_t)(bh * nchunks + c) * kMapBytes;
      *reinterpret_cast<float*>(map + kMcBytes + kNcBytes) = __expf(gC);
      bulk_s2g(map, mc_stage, kMcBytes);
      bulk_s2g(map + kMcBytes, nc_stage, kNcBytes);
      bulk_commit();
      bulk_wait_read<0>();
    }
    // x_last = phi(k_{T-1}) (last chunk, one warp)
    if (a.x_last && c == nchunks - 1 && warp == 4) {
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
  if (warp == 1) tmem_dealloc(tmem, 128);
}

}  // namespace

bool tc_falcon3a_applies(int dtype, int m, int dv, int C, int64_t BH, int64_t T) {
  return tc_path_applies(dtype, m, dv, C, BH, T) && m == 64;
}

cudaError_t launch_tc_falcon3a(const ChunkArgs& a, int window, int* err, cudaStream_t stream) {
  const int nchunks = (int)((a.T + k3C - 1) / k3C);
  CUtensorMap tm_k, tm_q, tm_v;
  if (!encode_rows_bf16(&tm_k, a.k, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, k3C) ||
      !encode_rows_bf16(&tm_q, a.q, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, k3C) ||
      !encode_rows_bf16(&tm_v, a.v, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, k3C))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_falcon3a_map_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kF3Smem);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch behind the preceding kernel (the map kernel
  // waits for it with griddepcontrol.wait before touching memory).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nchunks, (unsigned)a.BH);
  cfg.blockDim = dim3(k3Threads);
  cfg.dynamicSmemBytes = kF3Smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, tc_falcon3a_map_kernel, a, window, nchunks, err, tm_k, tm_q, tm_v);
  if (e != cudaSuccess) return e;
  return launch_tc_scan64(a, err, stream);
}

}  // namespace falcon
