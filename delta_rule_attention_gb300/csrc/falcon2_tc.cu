// Falcon-2 forward in chunk form on the tensor cores (bf16, m = d_v = 64,
// chunk 64).
//
// Page hyper.ai/fr/papers/2608.27763: the regression-family display of
// Section 3.1 with the per-column NLMS step sizes of Section 4.2.  Every value
// column j runs its own scalar-step delta rule on the shared write features,
//   r_{t,j} = v_{t,j} - s_j^T x_t,   s_j <- gamma_{j,t} s_j + eta_{j,t} x_t r_{t,j},
// so inside a chunk the written residuals u_{t,j} = eta_{j,t} r_{t,j} of
// column j solve a unit-lower system built from the shared Gram K = X X^T and
// the column's own decays (a batched per-column triangular solve with a
// shared Gram matrix).  With E_{t,j} the product of column j's gammas over the
// chunk's tokens up to t (E_{-1} = 1) and w_{l,j} = u_{l,j} / E_{l,j},
//   u_t = eta_t v_t - eta_t E_{t-1} ((X S)_t + sum_{l<t} K_{tl} w_l),
//   o_t = E_t ((Q S)_t + sum_{l<=t} <q_t, x_l> w_l),
//   S'  = E_C (S + X^T W)             (per column: E_C scales column j),
// which is the token recurrence unrolled over the chunk (w divides out the
// decays of the tokens up to l).  Every factor stays within fp32 range while
// a chunk's decay product is at least e^{-60} in every column; a chunk with a
// stronger decay (clamped gammas) runs the tokens one by one instead (exact,
// no factoring).
//
// One CTA per head runs the chunks in order (the per-column systems depend on
// the entering state), with three warp groups:
//   warps 0, 1  (solve; thread j owns column j): per chunk the tcgen05 MMA
//               S^T X^T gives (X S)^T with one column per TMEM lane; the solve
//               runs in four blocks of 16 rows: inside a block a thread runs
//               its column token by token (three dependent operations per
//               token); the blocks before it enter as one shared-Gram product
//               K_{b,<b} W_{<b} (warp-level bf16 MMAs).  The w rows, as bf16,
//               are the operand of the two MMAs that close the chunk: the state
//               increment W^T X, accumulated onto S^T in TMEM, and P0 W
//               (P0 = the causal part of Q X^T), accumulated onto Q S.  The
//               state S^T stays in TMEM in fp32.
//   warps 2, 3  (output): one chunk ahead, thread j runs column j's tokens in
//               order to form eta, gamma, the prefix products E and the
//               solve's per-token factors; then, for the current chunk,
//               thread t owns token row t: o_t = E_t (Q S + P0 W)_t from TMEM,
//               and one TMA store of the o tile.
//   warps 4..7  (prep, one chunk ahead): the k and q tiles (two-slot ring
//               refilled by the solve's issuing thread), phi's row scales, the
//               step-size denominators, the Gram MMA [K; Q] K^T on the raw bf16
//               rows with the scales applied afterwards in fp32.
// Every MMA reads the raw bf16 rows of k and q (exact inputs); phi's scales
// n_t enter in fp32, each once: the w rows carry the write features' scales
// (W' = n o w), the K tile its row scale only (K'_{tl} = n_t <k_t, k_l>, so
// that K' W' = K w), the rows of X S are scaled as they are read, and the
// output's Q S + P0 W' (raw q rows, P0 raw) is scaled by the q row's scale.
// The solve's per-chunk operands are double-buffered, so the prep of chunk
// c + 1 runs beside the chain of chunk c.
#include <cuda_bf16.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"
#include "tmap.cuh"

namespace falcon {

namespace {

using namespace tc;
using namespace tcu;

constexpr int kF2C = 64;         // chunk
constexpr int kF2Threads = 256;  // warps 0-1 solve, 2-3 output, 4-7 prep
constexpr int kF2Ring = 2;       // input-tile slots
// A chunk whose decay product in some column is below this runs token by
// token (e^{-60}: the factors 1/E and the w rows stay far inside fp32 range).
constexpr float kMinChunkDecay = 8.75651e-27f;

// Shared memory (bytes from a 1024-aligned base).
constexpr uint32_t kSlot = 2 * 8192;           // X | Q tiles (raw bf16 rows) of one chunk
constexpr uint32_t kRingOff = 0;               // kF2Ring slots
constexpr uint32_t kSopOff = kF2Ring * kSlot;  // S^T bf16, K-major rows j
constexpr uint32_t kWOff = kSopOff + 8192;     // W^T bf16, K-major rows j (tokens along K)
constexpr uint32_t kKbOff = kWOff + 8192;      // [2] K (strictly lower) bf16 rows t
constexpr uint32_t kPbOff = kKbOff + 2 * 8192; // P0 (causal Q X^T) bf16 rows t
constexpr uint32_t kOstOff = kPbOff + 8192;    // o tile for the TMA store
constexpr uint32_t kAOff = kOstOff + 8192;     // [2] eta_t E_{t-1} [j][t] fp32
constexpr uint32_t kFOff = kAOff + 2 * 16384;  // [2] 1 / E_t [j][t]
constexpr uint32_t kEvOff = kFOff + 2 * 16384; // [2] eta_t v_t [j][t]
constexpr uint32_t kE1Off = kEvOff + 2 * 16384;  // [2] E_t [t][j] (the output's scale)
constexpr uint32_t kKdOff = kE1Off + 2 * 16384;  // [2] K diagonal blocks fp32 [4][k][t]
constexpr int kTrsLd = 20;                     // fp32 row of the transpose scratch
constexpr uint32_t kTrsOff = kKdOff + 2 * 4096;  // [2 solve warps][32][kTrsLd]
constexpr uint32_t kSc2Off = kTrsOff + 2 * 32 * kTrsLd * 4;
// The MMAs with M = 128 read 64 rows past their operand: the state increment's
// A (W) reads the first K tile, the output's A (P0 as rows 64..127) starts at
// the second K tile; the lanes they fill are never read.
static_assert(kWOff + 8192 == kKbOff && kKbOff + 2 * 8192 == kPbOff, "operand layout");

struct F2cScalars {
  float nrm[2][128];  // phi's scale of row p of [X; Q], per chunk parity
  float lamr[2][64], inv[2][64];  // per token: lambda_t, 1 / (E + lambda + eps)
  float dC[2][64];    // E_C per column (the chunk's decay), per parity
  int flag[4];        // chunk c & 3 runs token by token
  uint64_t full[kF2Ring], xq[kF2Ring];
  uint64_t gdone, ydone, sdone, odone[2], obuf_free[2];
  uint64_t tok_ready[2], pre_ready[2], col_ready[2], solve_done[2], pb_ready;
  uint32_t tmem_base;
  int fail;
};
constexpr size_t kF2cSmem = kSc2Off + sizeof(F2cScalars) + 1024;
static_assert(kF2cSmem <= 232448, "Falcon-2 chunk kernel shared memory");

// TMEM columns: (X S)^T (lanes j), [X; Q] S + P0 W double-buffered (lanes t;
// rows 64..127 are the output), S^T (lanes j, fp32), the Gram (lanes t).
constexpr uint32_t kTmY = 0, kTmO = 64, kTmState = 192, kTmG = 256, kTmCols = 512;

// Element (j, t) of a [64][64] fp32 array whose 16-byte chunks are swizzled
// by j, so that a warp reading four consecutive tokens of 32 columns, or
// writing one column's 32 tokens, meets no bank conflict.  (The [t][j] array
// E uses the same map with the roles of t and j exchanged.)
__device__ __forceinline__ int jt(int j, int t) {
  return j * 64 + ((((t >> 2) ^ (j & 15))) << 2) + (t & 3);
}
__device__ __forceinline__ float4 jt4(const float* a, int j, int t4) {
  return *reinterpret_cast<const float4*>(a + jt(j, t4));
}

// Two 8 x 8 bf16 matrices (rows from lanes 0-7 and 8-15), not transposed: the
// mma.sync B fragment of an N x K row-major tile.
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(saddr)
               : "memory");
}

// Registers -> TMEM: 16 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Bounded wait for a role that is not on the chain: backs off between polls
// so that it takes few issue slots from the warps that are.
__device__ __forceinline__ bool mbar_wait_idle(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    __nanosleep(64);
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Row j of a K-major 128B-swizzled bf16 tile: the 16 values of chunk pair
// (2 q, 2 q + 1), i.e. columns 16 q .. 16 q + 15.
__device__ __forceinline__ void put_row16(unsigned char* tile, int j, int q, const float* v,
                                          float scale) {
  *reinterpret_cast<uint4*>(tile + sw_chunk(j, 2 * q)) = pack8(v, scale);
  *reinterpret_cast<uint4*>(tile + sw_chunk(j, 2 * q + 1)) = pack8(v + 8, scale);
}

// The contribution of the blocks before block b to its 16 rows, K_{b,<b}
// W_{<b} (one contraction over the 16 b tokens before the block), for this
// warp's 32 columns (warp-level bf16 MMAs, fp32 sums); returned per column:
// thread `lane` receives rows 0..15 of column 32 w + lane.  kb: the K tile
// (bf16 rows t), wt: the W^T tile (bf16 rows j), trs: the warp's transpose
// scratch (32 x kTrsLd floats).
__device__ __forceinline__ void horner16(uint32_t kb, uint32_t wt, int b, int w, float* trs,
                                         float (&r)[16]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  const int la = (lane & 7) + 8 * ((lane >> 3) & 1), ca = lane >> 4;
  float R[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) R[nt][e] = 0.f;
  for (int bp = 0; bp < b; ++bp) {
    uint32_t fa[4];
    ldsm_x4(fa, kb + sw_chunk(16 * b + la, 2 * bp + ca));
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      uint32_t fb[2];
      ldsm_x2(fb, wt + sw_chunk(32 * w + 8 * nt + (lane & 7), 2 * bp + ((lane >> 3) & 1)));
      mma16816(R[nt], fa, fb);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int c0 = 8 * nt + 2 * tq;
    trs[c0 * kTrsLd + g] = R[nt][0];
    trs[(c0 + 1) * kTrsLd + g] = R[nt][1];
    trs[c0 * kTrsLd + g + 8] = R[nt][2];
    trs[(c0 + 1) * kTrsLd + g + 8] = R[nt][3];
  }
  __syncwarp();
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const float4 x = *reinterpret_cast<const float4*>(trs + lane * kTrsLd + 4 * q4);
    r[4 * q4] = x.x;
    r[4 * q4 + 1] = x.y;
    r[4 * q4 + 2] = x.z;
    r[4 * q4 + 3] = x.w;
  }
  __syncwarp();
}

// One 64-element bf16 row of a 128B-swizzled tile times `scale`, into
// v[0..63] (fp32).
__device__ __forceinline__ void row_scaled(const unsigned char* tile, int r, float scale,
                                           float* v) {
  load_row_bf16(tile, r, v);
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] *= scale;
}

__global__ void __launch_bounds__(kF2Threads, 1)
    tc_falcon2_chunk_kernel(ChunkArgs a, int nch, int* err,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_o) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* const base = align1024(smem_raw);
  F2cScalars& sc = *reinterpret_cast<F2cScalars*>(base + kSc2Off);
  volatile int* fail = &sc.fail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bh = blockIdx.x;
  const int64_t T = a.T, rowbase = bh * T;
  auto arr = [&](uint32_t off, int par) { return reinterpret_cast<float*>(base + off) + par * 4096; };
  auto slot_addr = [&](int c) { return base + kRingOff + (c % kF2Ring) * kSlot; };
  // The k rows t0-1 .. t0+62 and q rows of chunk cc into its slot (rows
  // outside the sequence read as zero), and the chunk's gains, values and
  // ridges into L2 for the column pass.
  auto load_chunk = [&](int cc) {
    const int sl = cc % kF2Ring;
    unsigned char* dst = base + kRingOff + sl * kSlot;
    mbar_expect_tx(&sc.full[sl], 2 * 8192);
    tma_load_3d(dst, &tm_k, 0, cc * kF2C - 1, (int)bh, &sc.full[sl]);
    tma_load_3d(dst + 8192, &tm_q, 0, cc * kF2C, (int)bh, &sc.full[sl]);
    const int64_t t0 = (int64_t)cc * kF2C;
    const int nn = (int)min((int64_t)kF2C, T - t0);
    bulk_prefetch_l2(a.beta + (rowbase + t0) * 64, (uint32_t)nn * 256u);
    bulk_prefetch_l2(reinterpret_cast<const __nv_bfloat16*>(a.v) + (rowbase + t0) * 64,
                     (uint32_t)nn * 128u);
    const float* lp = a.lambda + rowbase + t0;  // (not 16-byte aligned in general)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(lp));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(lp + nn - 1));
    if (nn > 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(lp + 32));
  };

  if (warp == 0) tmem_alloc(&sc.tmem_base, kTmCols);
  if (tid == 32) {
    for (int i = 0; i < kF2Ring; ++i) {
      mbar_init(&sc.full[i], 1);
      mbar_init(&sc.xq[i], 1);
    }
    mbar_init(&sc.gdone, 1);
    mbar_init(&sc.ydone, 1);
    mbar_init(&sc.sdone, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sc.odone[i], 1);
      mbar_init(&sc.obuf_free[i], 2);
      mbar_init(&sc.tok_ready[i], 4);
      mbar_init(&sc.pre_ready[i], 4);
      mbar_init(&sc.col_ready[i], 2);
      mbar_init(&sc.solve_done[i], 2);
    }
    mbar_init(&sc.pb_ready, 2);
    for (int i = 0; i < 4; ++i) sc.flag[i] = 0;
    fence_mbar_init();
    sc.fail = 0;
  }
  // Launched behind the preceding kernel (programmatic dependent launch):
  // nothing is read or written before it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sc.tmem_base;
  const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);

  if (warp < 2) {
    // ======================= solve: thread j owns column j =======================
    const int j = tid, w = warp;
    float* trs = reinterpret_cast<float*>(base + kTrsOff) + w * 32 * kTrsLd;
    const uint32_t wt = smem_addr(base + kWOff);
    // The MMAs that open chunk c: (X S)^T (A = S^T, rows 64..127 past it land
    // in lanes nobody reads) and [X; Q] S into the output accumulator.
    auto open_chunk = [&](int c) {
      const int slot = c % kF2Ring;
      bool k2 = mbar_wait(&sc.xq[slot], (uint32_t)(c / kF2Ring) & 1u);
      if (c >= 2) k2 = k2 && mbar_wait(&sc.obuf_free[c & 1], (uint32_t)((c - 2) >> 1) & 1u);
      if (!k2) {
        *fail = 1;
        return;
      }
      tc_fence_after();
      const uint32_t xq = smem_addr(slot_addr(c));
      mma_k64(tmem + kTmY, smem_addr(base + kSopOff), false, 16, xq, false, 16,
              idesc_bf16(128, 64, false, false), false);
      mma_k64(tmem + kTmO + 64 * (c & 1), xq, false, 16, smem_addr(base + kSopOff), false, 16,
              idesc_bf16(128, 64, false, false), false);
      mma_commit(&sc.ydone);
    };
    // S0 into TMEM (fp32, lane j = column j) and the first state operand
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = a.S0 ? a.S0[(bh * 64 + 16 * q + i) * 64 + j] : 0.f;
      tmem_st16(tlane + kTmState + 16 * q, v);
      put_row16(base + kSopOff, j, q, v, 1.f);
    }
    tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    bool go = !named_sync_or(1, 64, false);
    if (go && tid == 0) open_chunk(0);
    for (int c = 0; go && c < nch; ++c) {
      const int slot = c % kF2Ring, par = c & 1;
      const unsigned char* xt = slot_addr(c);
      bool ok = mbar_wait(&sc.pre_ready[par], (uint32_t)(c >> 1) & 1u);
      ok = ok && mbar_wait(&sc.col_ready[par], (uint32_t)(c >> 1) & 1u);
      const bool tokenwise = sc.flag[c & 3] != 0;
      const float dC = sc.dC[par][j];  // read before this parity is released
      const float* A = arr(kAOff, par);
      const float* F = arr(kFOff, par);
      const float* EV = arr(kEvOff, par);
      ok = ok && mbar_wait(&sc.ydone, (uint32_t)c & 1u);
      tc_fence_after();
      if (!tokenwise) {
        const uint32_t kb = smem_addr(base + kKbOff + par * 8192);
        const float* KD = reinterpret_cast<const float*>(base + kKdOff) + par * 1024;
#pragma unroll 1
        for (int b = 0; b < 4; ++b) {
          float acc[16];
          tmem_ld16(tlane + kTmY + 16 * b, acc);
          {
            // phi's scales of the write features (the MMA read the raw k rows)
            const float* nx = sc.nrm[par] + 16 * b;
#pragma unroll
            for (int t = 0; t < 16; ++t) acc[t] *= nx[t];
          }
          if (b > 0) {
            float r[16];
            horner16(kb, wt, b, w, trs, r);
#pragma unroll
            for (int t = 0; t < 16; ++t) acc[t] += r[t];
          }
          float av[16], fv[16], ev[16];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float4 x = jt4(A, j, 16 * b + 4 * q4);
            const float4 y = jt4(F, j, 16 * b + 4 * q4);
            const float4 z = jt4(EV, j, 16 * b + 4 * q4);
            av[4 * q4] = x.x, av[4 * q4 + 1] = x.y, av[4 * q4 + 2] = x.z, av[4 * q4 + 3] = x.w;
            fv[4 * q4] = y.x, fv[4 * q4 + 1] = y.y, fv[4 * q4 + 2] = y.z, fv[4 * q4 + 3] = y.w;
            ev[4 * q4] = z.x, ev[4 * q4 + 1] = z.y, ev[4 * q4 + 2] = z.z, ev[4 * q4 + 3] = z.w;
          }
          const float* kd = KD + b * 256;
          float wv[16];
          // four tokens at a time: their Gram columns are loaded together, so
          // the shared-memory latency is paid once per four tokens
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            float kc[4][16];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int k = 4 * k4 + e;
#pragma unroll
              for (int q4 = (k + 1) >> 2; q4 < 4; ++q4) {
                const float4 x = *reinterpret_cast<const float4*>(kd + k * 16 + 4 * q4);
                kc[e][4 * q4] = x.x, kc[e][4 * q4 + 1] = x.y, kc[e][4 * q4 + 2] = x.z,
                    kc[e][4 * q4 + 3] = x.w;
              }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int k = 4 * k4 + e;
              const float u = fmaf(-av[k], acc[k], ev[k]);
              wv[k] = fv[k] * u;
#pragma unroll
              for (int t = k + 1; t < 16; ++t) acc[t] = fmaf(kc[e][t], wv[k], acc[t]);
            }
          }
          // the w rows of this block (bf16, with phi's scales: W') for the later
          // blocks and the MMAs
          put_row16(base + kWOff, j, b, wv, 1.f);
          __syncwarp();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc.solve_done[par]);
        fence_async_smem();
        tc_fence_before();
        if (named_sync_or(1, 64, !ok || *fail)) {
          *fail = 1;
          break;
        }
        if (tid == 0) {
          if (!mbar_wait(&sc.pb_ready, (uint32_t)c & 1u)) {
            *fail = 1;
          } else {
            tc_fence_after();
            // S^T += W^T X (A = W^T K-major, B = X MN-major); Q S += P0 W
            mma_k64(tmem + kTmState, wt, false, 16, smem_addr(xt), true, 8192,
                    idesc_bf16(128, 64, false, true), true);
            mma_k64(tmem + kTmO + 64 * par, smem_addr(base + kKbOff + 8192), false, 16, wt,
                    false, 16, idesc_bf16(128, 64, false, false), true);
            mma_commit(&sc.sdone);
            mma_commit(&sc.odone[par]);
          }
        }
        ok = mbar_wait(&sc.sdone, (uint32_t)c & 1u);
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float sv[16];
          tmem_ld16(tlane + kTmState + 16 * q, sv);
#pragma unroll
          for (int i = 0; i < 16; ++i) sv[i] *= dC;
          tmem_st16(tlane + kTmState + 16 * q, sv);
          put_row16(base + kSopOff, j, q, sv, 1.f);
        }
      } else {
        // Token by token (a decay too strong to factor), from the inputs.
        const int64_t t0 = (int64_t)c * kF2C;
        const int n = (int)min((int64_t)kF2C, T - t0);
        float s[64];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tlane + kTmState + 16 * q, s + 16 * q);
        __nv_bfloat16* og = reinterpret_cast<__nv_bfloat16*>(a.o) + (rowbase + t0) * 64 + j;
        const __nv_bfloat16* vg =
            reinterpret_cast<const __nv_bfloat16*>(a.v) + (rowbase + t0) * 64 + j;
        const float* bg = a.beta + (rowbase + t0) * 64 + j;
        const float eg = a.eps_gamma;
        for (int t = 0; t < n; ++t) {
          const float eta = bg[(int64_t)t * 64] * sc.inv[par][t];
          const float al = eta * sc.lamr[par][t];
          const float gam = al >= 1.f - eg ? eg : 1.f - al;
          const float etav = eta * __bfloat162float(vg[(int64_t)t * 64]);
          float x[64];
          row_scaled(xt, t, sc.nrm[par][t], x);
          float d8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 64; ++i) d8[i & 7] = fmaf(s[i], x[i], d8[i & 7]);
          const float d = ((d8[0] + d8[1]) + (d8[2] + d8[3])) + ((d8[4] + d8[5]) + (d8[6] + d8[7]));
          const float u = fmaf(-eta, d, etav);
#pragma unroll
          for (int i = 0; i < 64; ++i) s[i] = fmaf(u, x[i], gam * s[i]);
          row_scaled(xt + 8192, t, sc.nrm[par][64 + t], x);
#pragma unroll
          for (int i = 0; i < 8; ++i) d8[i] = 0.f;
#pragma unroll
          for (int i = 0; i < 64; ++i) d8[i & 7] = fmaf(s[i], x[i], d8[i & 7]);
          og[(int64_t)t * 64] = __float2bfloat16_rn(
              ((d8[0] + d8[1]) + (d8[2] + d8[3])) + ((d8[4] + d8[5]) + (d8[6] + d8[7])));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc.solve_done[par]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          tmem_st16(tlane + kTmState + 16 * q, s + 16 * q);
          put_row16(base + kSopOff, j, q, s + 16 * q, 1.f);
        }
        if (named_sync_or(1, 64, !ok || *fail)) {
          *fail = 1;
          break;
        }
        // no MMA closes this chunk: keep the barriers' phases in step
        if (tid == 0) {
          if (!mbar_wait(&sc.pb_ready, (uint32_t)c & 1u)) *fail = 1;
          mbar_arrive(&sc.sdone);
          mbar_arrive(&sc.odone[par]);
        }
        ok = ok && mbar_wait(&sc.sdone, (uint32_t)c & 1u);
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      if (named_sync_or(1, 64, !ok || *fail)) {
        *fail = 1;
        break;
      }
      if (tid == 0) {
        if (c + 1 < nch) open_chunk(c + 1);
        // the slot of chunk c is free: chunk c + 2 into it
        if (c + 2 < nch) load_chunk(c + 2);
      }
    }
    if (!*fail) {
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float sv[16];
        tmem_ld16(tlane + kTmState + 16 * q, sv);
#pragma unroll
        for (int i = 0; i < 16; ++i) a.S_out[(bh * 64 + 16 * q + i) * 64 + j] = sv[i];
      }
    }
  } else if (warp < 4) {
    // ======================= output =======================
    const int me = tid - 64;  // column (the pass ahead) and token row (the output)
    unsigned char* ost = base + kOstOff;
    float nq[2] = {0.f, 0.f};  // phi's scale of q row `me`, per chunk parity
    // Column pass of chunk cc: eta, gamma and the prefix products E of column
    // j = me token by token; the solve's factors A = eta E_{t-1}, F = n_t / E_t,
    // eta v, the output's E, and the chunk's decay E_C (dC).
    auto column_pass = [&](int cc) -> bool {
      const int pp = cc & 1;
      bool ok = mbar_wait_idle(&sc.tok_ready[pp], (uint32_t)(cc >> 1) & 1u);
      // this parity's buffers were last read by the solve of chunk cc - 2
      if (cc >= 2) ok = ok && mbar_wait_idle(&sc.solve_done[pp], (uint32_t)((cc - 2) >> 1) & 1u);
      float* A = arr(kAOff, pp);
      float* F = arr(kFOff, pp);
      float* EV = arr(kEvOff, pp);
      float* E1 = arr(kE1Off, pp);
      const int j = me;
      const float eg = a.eps_gamma;
      nq[pp] = sc.nrm[pp][64 + me];
      // the prep staged the column's gains in A and values in EV ([j][t]);
      // they are overwritten in place with the solve's factors
      float E = 1.f;  // E_{t-1}
#pragma unroll
      for (int t4 = 0; t4 < 64; t4 += 4) {
        const float4 b4 = jt4(A, j, t4), vv4 = jt4(EV, j, t4);
        const float be[4] = {b4.x, b4.y, b4.z, b4.w}, ve[4] = {vv4.x, vv4.y, vv4.z, vv4.w};
        float a4[4], f4[4], v4[4], e4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = t4 + e;
          const float eta = be[e] * sc.inv[pp][t];
          const float al = eta * sc.lamr[pp][t];
          const float gam = al >= 1.f - eg ? eg : 1.f - al;
          const float En = E * gam;
          a4[e] = eta * E;
          f4[e] = __fdividef(sc.nrm[pp][t], En);  // (E_t >= e^{-60} on the factored path)
          v4[e] = eta * ve[e];
          e4[e] = En;
          E = En;
        }
        *reinterpret_cast<float4*>(A + jt(j, t4)) = make_float4(a4[0], a4[1], a4[2], a4[3]);
        *reinterpret_cast<float4*>(F + jt(j, t4)) = make_float4(f4[0], f4[1], f4[2], f4[3]);
        *reinterpret_cast<float4*>(EV + jt(j, t4)) = make_float4(v4[0], v4[1], v4[2], v4[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e) E1[jt(t4 + e, j)] = e4[e];
      }
      sc.dC[pp][j] = E;
      // a column whose decay over the chunk is too strong to factor sends the
      // whole chunk token by token
      const bool weak = !(E >= kMinChunkDecay);
      const bool any = named_sync_or(2, 64, weak);
      if (me == 0) sc.flag[cc & 3] = any ? 1 : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc.col_ready[pp]);
      return ok;
    };
    bool ok = nch > 0 ? column_pass(0) : true;
    for (int c = 0; c < nch; ++c) {
      const int par = c & 1, t = me;
      if (c + 1 < nch) ok = column_pass(c + 1) && ok;
      if (tid == 64) bulk_wait_read<0>();  // the previous o store has read the tile
      if (named_sync_or(2, 64, !ok || *fail)) {
        *fail = 1;
        break;
      }
      ok = mbar_wait_idle(&sc.odone[par], (uint32_t)(c >> 1) & 1u);
      const bool tokenwise = sc.flag[c & 3] != 0;
      if (!tokenwise) {
        tc_fence_after();
        float d[64];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tlane + kTmO + 64 * par + 16 * q, d + 16 * q);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc.obuf_free[par]);
        // o_t = E_t n_q (Q S + P0 W')_t (raw q rows and P0), E in [t][j]
        const float* E1 = arr(kE1Off, par);
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 e = *reinterpret_cast<const float4*>(E1 + jt(t, 4 * q4));
          d[4 * q4] *= nq[par] * e.x, d[4 * q4 + 1] *= nq[par] * e.y,
              d[4 * q4 + 2] *= nq[par] * e.z, d[4 * q4 + 3] *= nq[par] * e.w;
        }
        store_row_bf16(ost, t, d);
        fence_async_smem();
        if (named_sync_or(2, 64, !ok || *fail)) {
          *fail = 1;
          break;
        }
        if (tid == 64) {
          tma_store_3d(&tm_o, ost, 0, c * kF2C, (int)bh);
          bulk_commit();
        }
      } else {
        // the solve warps wrote this chunk's o rows themselves
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc.obuf_free[par]);
        if (!ok) *fail = 1;
      }
    }
    if (tid == 64) bulk_wait<0>();
  } else {
    // ======================= prep: one chunk ahead =======================
    const int p = tid - 128;  // row of [X; Q] (features, Gram rows)
    const int tt = p & 63;
    const bool issuer = p == 0;
    if (issuer)
      for (int cc = 0; cc < kF2Ring && cc < nch; ++cc) load_chunk(cc);
    for (int c = 0; c < nch; ++c) {
      const int slot = c % kF2Ring, par = c & 1;
      const int64_t t0 = (int64_t)c * kF2C;
      const int n = (int)min((int64_t)kF2C, T - t0);
      unsigned char* xt = base + kRingOff + slot * kSlot;  // X, then Q at +8 KB
      bool ok = true;
      const float lam_t = (p < 64 && p < n) ? a.lambda[rowbase + t0 + p] : 0.f;
      // gains and values of token tt, columns 32 hh .. 32 hh + 31 (16-byte loads),
      // staged transposed for the column pass (zero past the sequence)
      const int hh = p >> 6;
      float4 bet[8];
      uint4 vraw[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) bet[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 4; ++i) vraw[i] = make_uint4(0u, 0u, 0u, 0u);
      if (tt < n) {
        const float4* src =
            reinterpret_cast<const float4*>(a.beta + (rowbase + t0 + tt) * 64 + 32 * hh);
#pragma unroll
        for (int i = 0; i < 8; ++i) bet[i] = src[i];
        const uint4* vs = reinterpret_cast<const uint4*>(
            reinterpret_cast<const __nv_bfloat16*>(a.v) + (rowbase + t0 + tt) * 64 + 32 * hh);
#pragma unroll
        for (int i = 0; i < 4; ++i) vraw[i] = vs[i];
      }
      ok = ok && mbar_wait_idle(&sc.full[slot], (uint32_t)(c / kF2Ring) & 1u);
      // this parity's buffers (phi's scales, the denominators, the Gram tiles)
      // were last read by the solve of chunk c - 2
      if (c >= 2) ok = ok && mbar_wait_idle(&sc.solve_done[par], (uint32_t)((c - 2) >> 1) & 1u);
      const bool carried = c == 0 && p == 0 && a.x_prev != nullptr;
      if (c == 0 && a.x_prev != nullptr && p < 8) {
        // x_1 = x_prev (already phi-mapped) in row 0 of the X tile
        float v8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v8[e] = a.x_prev[bh * 64 + 8 * p + e];
        *reinterpret_cast<uint4*>(xt + (p << 4)) = pack8(v8, 1.f);  // row 0: no swizzle shift
      }
      fence_async_smem();
      if (named_sync_or(3, 128, !ok || *fail)) {
        *fail = 1;
        break;
      }
      if (issuer) {
        tc_fence_after();
        // Gram on the raw rows: [K; Q] K^T (phi's scales enter at the readback)
        mma_k64(tmem + kTmG, smem_addr(xt), false, 16, smem_addr(xt), false, 16,
                idesc_bf16(128, 64, false, false), false);
        mma_commit(&sc.gdone);
        mbar_arrive(&sc.xq[slot]);  // the tiles are in place for the chain's MMAs
      }
      // phi's scale of row p (p < 64: x_p = phi(k_{t0+p-1}); else phi(q_{t0+p-64}))
      // and the token's step-size denominator
      float nr;
      {
        float row[64];
        load_row_bf16(xt, p, row);  // X and Q tiles are contiguous: row p of [X; Q]
        float ss = 0.f;
        if (carried) {
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            const float x = a.x_prev[bh * 64 + i];
            ss = fmaf(x, x, ss);
          }
        } else {
          float q8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 64; ++i) q8[i & 7] = fmaf(row[i], row[i], q8[i & 7]);
          ss = ((q8[0] + q8[1]) + (q8[2] + q8[3])) + ((q8[4] + q8[5]) + (q8[6] + q8[7]));
        }
        nr = carried ? 1.f : phi_scale(ss, 64, a.phi);
        sc.nrm[par][p] = nr;
        if (p < 64) {
          const float E = ss * nr * nr;
          const float lam = ridge_of(lam_t, E, a.ridge);
          const float den = E + lam + a.eps;
          const bool sentinel = t0 + p == 0 && a.x_prev == nullptr;
          sc.lamr[par][p] = lam;
          sc.inv[par][p] = (!sentinel && p < n && den > 0.f) ? 1.f / den : 0.f;
        }
      }
      {
        float* Ab = arr(kAOff, par);
        float* EVb = arr(kEvOff, par);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float bb[4] = {bet[i].x, bet[i].y, bet[i].z, bet[i].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) Ab[jt(32 * hh + 4 * i + e, tt)] = bb[e];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162* h2v = reinterpret_cast<const __nv_bfloat162*>(&vraw[i]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h2v[e]);
            EVb[jt(32 * hh + 8 * i + 2 * e, tt)] = f.x;
            EVb[jt(32 * hh + 8 * i + 2 * e + 1, tt)] = f.y;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc.tok_ready[par]);
      // Gram readback: rows 0..63 are K' = n_t <k_t, k_l> (l < t; the column
      // scale n_l rides on W'), rows 64..127 the raw causal <q_t, k_l> (l <= t)
      float d[64];
      {
        ok = ok && mbar_wait_idle(&sc.gdone, (uint32_t)c & 1u);
        tc_fence_after();
        tmem_ld32(tlane + kTmG, d);
        tmem_ld32(tlane + kTmG + 32, d + 32);
        const bool krow = p < 64;
        const float rs = krow ? nr : 1.f;
#pragma unroll
        for (int l = 0; l < 64; ++l) {
          const bool keep = krow ? (l < tt) : (l <= tt);
          d[l] = keep ? d[l] * rs : 0.f;
        }
        if (krow) {
          unsigned char* kbt = base + kKbOff + par * 8192;
#pragma unroll
          for (int q = 0; q < 4; ++q) put_row16(kbt, tt, q, d + 16 * q, 1.f);
          float* dg = reinterpret_cast<float*>(base + kKdOff) + par * 1024 + (tt >> 4) * 256 +
                      (tt & 15);
#pragma unroll
          for (int bb = 0; bb < 4; ++bb)
            if (bb == (tt >> 4))
#pragma unroll
              for (int k = 0; k < 16; ++k) dg[k * 16] = d[16 * bb + k];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc.pre_ready[par]);
      // The P0 tile (single buffer: the output MMA of chunk c - 1 has completed)
      if (p >= 64) {
        if (c >= 1)
          ok = ok && mbar_wait_idle(&sc.odone[(c - 1) & 1], (uint32_t)((c - 1) >> 1) & 1u);
#pragma unroll
        for (int q = 0; q < 4; ++q) put_row16(base + kPbOff, tt, q, d + 16 * q, 1.f);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc.pb_ready);
      }
      if (!ok) *fail = 1;
    }
    // x_last = phi(k_{T-1})
    if (a.x_last && warp == 4) {
      const __nv_bfloat16* kl =
          reinterpret_cast<const __nv_bfloat16*>(a.k) + (rowbase + T - 1) * 64;
      const float u0 = __bfloat162float(kl[lane]), u1 = __bfloat162float(kl[lane + 32]);
      const float s2 = phi_scale(warp_sum(u0 * u0 + u1 * u1), 64, a.phi);
      a.x_last[bh * 64 + lane] = u0 * s2;
      a.x_last[bh * 64 + lane + 32] = u1 * s2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*fail && tid == 0) flag_error(err);
  if (warp == 0) tmem_dealloc(tmem, kTmCols);
}

}  // namespace

bool tc_falcon2_applies(int dtype, int m, int dv, int C, int64_t BH, int64_t T) {
  return tc_path_applies(dtype, m, dv, C, BH, T) && m == 64;
}

cudaError_t launch_tc_falcon2(const ChunkArgs& a, int* err, cudaStream_t stream) {
  const int nch = (int)((a.T + kF2C - 1) / kF2C);
  CUtensorMap tm_k, tm_q, tm_o;
  if (!encode_rows_bf16(&tm_k, a.k, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kF2C) ||
      !encode_rows_bf16(&tm_q, a.q, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kF2C) ||
      !encode_rows_bf16(&tm_o, a.o, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kF2C))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_falcon2_chunk_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kF2cSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.BH);
  cfg.blockDim = dim3(kF2Threads);
  cfg.dynamicSmemBytes = kF2cSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_falcon2_chunk_kernel, a, nch, err, tm_k, tm_q, tm_o);
}

}  // namespace falcon
