// Falcon-2 forward in chunk form on the tensor cores (bf16, m = d_v = 64,
// chunk 64).
//
// Page hyper.ai/fr/papers/2608.27763: the regression-family display of
// Section 3.1 with the per-column NLMS step sizes of Section 4.2.  Every value
// column j runs its own scalar-step delta rule on the shared write features,
//   r_{t,j} = v_{t,j} - s_j^T x_t,   s_j <- gamma_{j,t} s_j + eta_{j,t} x_t r_{t,j},
// so inside a chunk the written residuals u_{t,j} = eta_{j,t} r_{t,j} of
// column j solve a unit-lower system built from the shared Gram K = X X^T and
// the column's own decays (the "batched per-channel triangular solve with a
// shared Gram matrix").  With e^{G_{j,i}} the product of the column's gammas
// over the chunk's tokens up to i, and the accumulator
//   acc^{(i)}_t = e^{G_i} (X S)_t + sum_{l<=i} e^{G_i - G_l} K_{tl} u_l,
// the residual of row t is v_t - acc^{(t-1)}_t and acc^{(i)} = gamma_i
// acc^{(i-1)} + K_{.,i} u_i: only products of gammas, never an exponential,
// so strong and clamped decays cannot overflow anything.  The chunk's 64 rows
// go in four blocks of 16: inside a block the accumulators run token by token
// (one thread per column, fp32 registers); the blocks before it enter through
// the shared matrices, sum_{b'<b} (decay) K_{b,b'} U~^{[b']}, combined in
// Horner order with the block decays (warp-level bf16 MMAs, fp32 sums).  The
// output and the state leaving the chunk are
//   o_{t,j}  = e^{G_t} (Q S)_{t,j} + sum_{l<=t} e^{G_t - G_l} <q_t, x_l> u_{l,j},
//   S'_{:,j} = e^{G_C} S_{:,j} + sum_l x_l e^{G_C - G_l} u_{l,j}.
//
// One CTA per head runs the chunks in order (the per-column systems depend on
// the entering state), with three warp groups:
//   warps 0, 1  (solve; thread j owns column j): the state column s_j in fp32
//               registers; per chunk the tcgen05 MMA [S^T; S^T] [X; Q]^T gives
//               (X S)^T and (Q S)^T with one column per TMEM lane, the blocked
//               solve, then the MMA (e^{G_C - G} o U)^T X for the state
//               increment.  These two MMAs and the solve are the sequential
//               chain.
//   warps 2, 3  (output; column j): the output rows block by block, behind the
//               solve, and one TMA store of the o tile per chunk.
//   warps 4..7  (prep, one chunk ahead): the k, q, v tiles by TMA (three-slot
//               ring), the Gram MMA [K; Q] K^T on the raw bf16 rows with phi's
//               scales applied afterwards in fp32, the features phi(k), phi(q)
//               in place, and per (token, column) eta, gamma and eta * v.
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
constexpr int kF2Ring = 3;       // input-tile slots

// Shared memory (bytes from a 1024-aligned base).
constexpr uint32_t kSlot = 3 * 8192;            // X | Q | V tiles of one chunk
constexpr uint32_t kRingOff = 0;                // kF2Ring slots
constexpr uint32_t kSopOff = kF2Ring * kSlot;   // [S^T; S^T] bf16, K-major (16 KB)
constexpr uint32_t kDecuOff = kSopOff + 16384;  // (e^{G_C-G} o U)^T bf16, K-major (8 KB);
                                                // the MMA's rows 64..127 read the KB
                                                // tile after it (lanes nobody reads)
constexpr uint32_t kKbOff = kDecuOff + 8192;    // K as bf16, 128B-swizzled rows
constexpr uint32_t kPbOff = kKbOff + 8192;      // P0 = Q X^T as bf16
constexpr uint32_t kOstOff = kPbOff + 8192;     // o tile for the TMA store
constexpr uint32_t kEtaOff = kOstOff + 8192;    // eta [j][t] fp32 (swizzled chunks)
constexpr uint32_t kGamOff = kEtaOff + 16384;   // gamma [j][t]
constexpr uint32_t kEtavOff = kGamOff + 16384;  // eta * v [j][t]
constexpr uint32_t kUOff = kEtavOff + 16384;    // u [j][t]
constexpr uint32_t kUtOff = kUOff + 16384;      // U~ blocks, bf16 [2][4][64 j][16 l]
constexpr uint32_t kKdOff = kUtOff + 16384;     // K diagonal blocks fp32 [4][k][t]
constexpr uint32_t kPdOff = kKdOff + 4096;      // P0 diagonal blocks fp32 [4][i][t]
constexpr int kTrsLd = 20;                      // fp32 row of the transpose scratch
constexpr uint32_t kTrsOff = kPdOff + 4096;     // [solve, output][2 warps][32][kTrsLd]
constexpr uint32_t kDblkOff = kTrsOff + 2 * 2 * 32 * kTrsLd * 4;  // [2][4][64] fp32
constexpr uint32_t kSc2Off = kDblkOff + 2 * 4 * 64 * 4;

struct F2cScalars {
  float nrm[128];  // phi's scale of row p of [X; Q]
  float E[64], lamr[64], inv[64];
  uint64_t full[kF2Ring], empty[kF2Ring], xq[kF2Ring];
  uint64_t gdone, ydone[2], sdone, ybuf_free[2];
  uint64_t pre_ready, solve_blk[4], out_blk[4], decu_done;
  uint32_t tmem_base;
  int fail;
};
constexpr size_t kF2cSmem = kSc2Off + sizeof(F2cScalars) + 1024;
static_assert(kF2cSmem <= 232448, "Falcon-2 chunk kernel shared memory");
static_assert(kDecuOff + 8192 == kKbOff, "MMA_S reads rows 64..127 from the KB tile");

// TMEM columns: the (X S | Q S)^T accumulator, double-buffered (128 columns
// each), the state increment (64) and the Gram (64).
constexpr uint32_t kTmY = 0, kTmS = 256, kTmG = 320, kTmCols = 512;

// Element (j, t) of a [64][64] fp32 array whose 16-byte chunks are swizzled
// by j, so that a warp reading four consecutive tokens of 32 columns, or
// writing one column's 32 tokens, meets no bank conflict.
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

// Byte offset of U~ block b (buffer yb), column j, 16-byte chunk c.
__device__ __forceinline__ uint32_t ut_off(int yb, int b, int j, int c) {
  return (uint32_t)(yb * 8192 + b * 2048) + dblk_chunk(j, c);
}

// The contribution of the blocks before block b to the 16 rows of block b,
//   R = sum_{b'<b} (prod of the block decays after b') M_{b,b'} U~^{[b']},
// for this warp's 32 columns (Horner order over b'), with M the bf16 tile
// `mt` (K or P0, 128B-swizzled rows); returned per column: thread `lane`
// receives rows 0..15 of column 32 w + lane in r.  trs: the warp's transpose
// scratch (32 x kTrsLd floats).
__device__ __forceinline__ void horner16(const unsigned char* base, uint32_t mt_off, int yb,
                                         int b, int w, const float* dblk, float* trs,
                                         float (&r)[16]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, tq = lane & 3;
  const int la = (lane & 7) + 8 * ((lane >> 3) & 1), ca = lane >> 4;
  float R[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) R[nt][e] = 0.f;
  const uint32_t mbase = smem_addr(base + mt_off);
  const uint32_t ubase = smem_addr(base + kUtOff);
  for (int bp = 0; bp < b; ++bp) {
    uint32_t fa[4];
    ldsm_x4(fa, mbase + sw_chunk(16 * b + la, 2 * bp + ca));
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = 32 * w + 8 * nt + 2 * tq;
      const float d0 = dblk[bp * 64 + col], d1 = dblk[bp * 64 + col + 1];
      R[nt][0] *= d0;
      R[nt][1] *= d1;
      R[nt][2] *= d0;
      R[nt][3] *= d1;
      uint32_t fb[2];
      ldsm_x2(fb, ubase + ut_off(yb, bp, 32 * w + 8 * nt + (lane & 7), (lane >> 3) & 1));
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

// A 64-value fp32 row as bf16 into row r of a 128B-swizzled K-major tile.
__device__ __forceinline__ void put_row64(unsigned char* tile, int r, const float* v) {
  store_row_bf16(tile, r, v);
}

__global__ void __launch_bounds__(kF2Threads, 1)
    tc_falcon2_chunk_kernel(ChunkArgs a, int nch, int* err,
                            const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ CUtensorMap tm_o) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* const base = align1024(smem_raw);
  F2cScalars& sc = *reinterpret_cast<F2cScalars*>(base + kSc2Off);
  volatile int* fail = &sc.fail;
  float* const ETA = reinterpret_cast<float*>(base + kEtaOff);
  float* const GAM = reinterpret_cast<float*>(base + kGamOff);
  float* const ETAV = reinterpret_cast<float*>(base + kEtavOff);
  float* const UB = reinterpret_cast<float*>(base + kUOff);
  float* const KD = reinterpret_cast<float*>(base + kKdOff);
  float* const PD = reinterpret_cast<float*>(base + kPdOff);
  float* const DBLK = reinterpret_cast<float*>(base + kDblkOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t bh = blockIdx.x;
  const int64_t T = a.T, rowbase = bh * T;

  if (warp == 0) tmem_alloc(&sc.tmem_base, kTmCols);
  if (tid == 32) {
    for (int i = 0; i < kF2Ring; ++i) {
      mbar_init(&sc.full[i], 1);
      mbar_init(&sc.empty[i], 1);
      mbar_init(&sc.xq[i], 1);
    }
    mbar_init(&sc.gdone, 1);
    mbar_init(&sc.ydone[0], 1);
    mbar_init(&sc.ydone[1], 1);
    mbar_init(&sc.sdone, 1);
    mbar_init(&sc.ybuf_free[0], 2);
    mbar_init(&sc.ybuf_free[1], 2);
    mbar_init(&sc.pre_ready, 4);
    for (int b = 0; b < 4; ++b) {
      mbar_init(&sc.solve_blk[b], 2);
      mbar_init(&sc.out_blk[b], 2);
    }
    mbar_init(&sc.decu_done, 2);
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
    float s[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) s[i] = a.S0 ? a.S0[(bh * 64 + i) * 64 + j] : 0.f;
    for (int c = 0; c < nch; ++c) {
      const int slot = c % kF2Ring, yb = c & 1;
      bool ok = true;
      // state operand: rows j and 64 + j of [S^T; S^T]
      put_row64(base + kSopOff, j, s);
      put_row64(base + kSopOff, 64 + j, s);
      fence_async_smem();
      tc_fence_before();
      if (named_sync_or(1, 64, *fail)) break;
      if (tid == 0) {
        bool k2 = mbar_wait(&sc.xq[slot], (uint32_t)(c / kF2Ring) & 1u);
        if (c >= 2) k2 = k2 && mbar_wait(&sc.ybuf_free[yb], (uint32_t)((c - 2) >> 1) & 1u);
        if (!k2) {
          *fail = 1;
        } else {
          tc_fence_after();
          // (X S | Q S)^T: A = [S^T; S^T] (K-major), B = [X; Q] (K-major, N = 128)
          mma_k64(tmem + kTmY + 128 * yb, smem_addr(base + kSopOff), false, 16,
                  smem_addr(base + kRingOff + slot * kSlot), false, 16,
                  idesc_bf16(128, 128, false, false), false);
          mma_commit(&sc.ydone[yb]);
        }
      }
      ok = ok && mbar_wait(&sc.pre_ready, (uint32_t)c & 1u);
      ok = ok && mbar_wait(&sc.ydone[yb], (uint32_t)(c >> 1) & 1u);
      tc_fence_after();
      float pc = 1.f;  // product of gamma over the blocks before b
      float u[16];
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        float acc[16];
        tmem_ld16(tlane + kTmY + 128 * yb + 16 * b, acc);
        if (b > 0) {
          float r[16];
          horner16(base, kKbOff, yb, b, w, DBLK + yb * 256, trs, r);
#pragma unroll
          for (int t = 0; t < 16; ++t) acc[t] = fmaf(pc, acc[t], r[t]);
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) acc[t] *= pc;
        }
        float eta[16], etav[16], gam[16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 e = jt4(ETA, j, 16 * b + 4 * q4);
          const float4 ev = jt4(ETAV, j, 16 * b + 4 * q4);
          const float4 g = jt4(GAM, j, 16 * b + 4 * q4);
          eta[4 * q4] = e.x, eta[4 * q4 + 1] = e.y, eta[4 * q4 + 2] = e.z, eta[4 * q4 + 3] = e.w;
          etav[4 * q4] = ev.x, etav[4 * q4 + 1] = ev.y, etav[4 * q4 + 2] = ev.z,
                    etav[4 * q4 + 3] = ev.w;
          gam[4 * q4] = g.x, gam[4 * q4 + 1] = g.y, gam[4 * q4 + 2] = g.z, gam[4 * q4 + 3] = g.w;
        }
        const float* kd = KD + b * 256;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          u[k] = fmaf(-eta[k], acc[k], etav[k]);
          float kc[16];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float4 x = *reinterpret_cast<const float4*>(kd + k * 16 + 4 * q4);
            kc[4 * q4] = x.x, kc[4 * q4 + 1] = x.y, kc[4 * q4 + 2] = x.z, kc[4 * q4 + 3] = x.w;
          }
#pragma unroll
          for (int t = k + 1; t < 16; ++t) acc[t] = fmaf(kc[t], u[k], gam[k] * acc[t]);
        }
        // U~ (u decayed to the block's end) and the block decay
        float d = 1.f;
        float ut[16];
#pragma unroll
        for (int k = 15; k >= 0; --k) {
          ut[k] = d * u[k];
          d *= gam[k];
        }
        // u of this block is read by the output warps of the previous chunk
        // until they are past block b.
        if (c > 0) ok = ok && mbar_wait(&sc.out_blk[b], (uint32_t)(c - 1) & 1u);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          *reinterpret_cast<float4*>(UB + jt(j, 16 * b + 4 * q4)) =
              make_float4(u[4 * q4], u[4 * q4 + 1], u[4 * q4 + 2], u[4 * q4 + 3]);
        *reinterpret_cast<uint4*>(base + kUtOff + ut_off(yb, b, j, 0)) = pack8(ut, 1.f);
        *reinterpret_cast<uint4*>(base + kUtOff + ut_off(yb, b, j, 1)) = pack8(ut + 8, 1.f);
        DBLK[yb * 256 + b * 64 + j] = d;
        pc *= d;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc.solve_blk[b]);
      }
      // (e^{G_C - G_l} u_l) for the state increment; e^{G_C} = pc
      {
        float dv[64];
        float d = 1.f;
#pragma unroll
        for (int q4 = 15; q4 >= 0; --q4) {
          const float4 uu = jt4(UB, j, 4 * q4);
          const float4 g = jt4(GAM, j, 4 * q4);
          dv[4 * q4 + 3] = d * uu.w;
          d *= g.w;
          dv[4 * q4 + 2] = d * uu.z;
          d *= g.z;
          dv[4 * q4 + 1] = d * uu.y;
          d *= g.y;
          dv[4 * q4] = d * uu.x;
          d *= g.x;
        }
        put_row64(base + kDecuOff, j, dv);
      }
      fence_async_smem();
      tc_fence_before();
      if (named_sync_or(1, 64, !ok || *fail)) {
        *fail = 1;
        break;
      }
      if (lane == 0) mbar_arrive(&sc.decu_done);
      if (tid == 0) {
        tc_fence_after();
        // increment^T = (e^{G_C - G} o U)^T X: A K-major (rows j), B = X MN-major
        mma_k64(tmem + kTmS, smem_addr(base + kDecuOff), false, 16,
                smem_addr(base + kRingOff + slot * kSlot), true, 8192,
                idesc_bf16(128, 64, false, true), false);
        mma_commit(&sc.sdone);
      }
      ok = mbar_wait(&sc.sdone, (uint32_t)c & 1u);
      tc_fence_after();
      if (tid == 0) mbar_arrive(&sc.empty[slot]);  // X, Q, V of chunk c are no longer read
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float inc[16];
        tmem_ld16(tlane + kTmS + 16 * q, inc);
#pragma unroll
        for (int i = 0; i < 16; ++i) s[16 * q + i] = fmaf(pc, s[16 * q + i], inc[i]);
      }
      if (!ok) *fail = 1;
    }
    if (!*fail) {
#pragma unroll
      for (int i = 0; i < 64; ++i) a.S_out[(bh * 64 + i) * 64 + j] = s[i];
    }
  } else if (warp < 4) {
    // ======================= output: thread owns column j =======================
    const int j = tid - 64, w = warp - 2;
    float* trs = reinterpret_cast<float*>(base + kTrsOff) + (2 + w) * 32 * kTrsLd;
    unsigned char* ost = base + kOstOff;
    for (int c = 0; c < nch; ++c) {
      const int yb = c & 1;
      bool ok = true;
      if (tid == 64) bulk_wait_read<0>();  // the previous o store has read the tile
      if (named_sync_or(2, 64, *fail)) break;
      ok = ok && mbar_wait(&sc.pre_ready, (uint32_t)c & 1u);
      ok = ok && mbar_wait(&sc.ydone[yb], (uint32_t)(c >> 1) & 1u);
      tc_fence_after();
      float pc = 1.f;
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
        float ao[16];
        tmem_ld16(tlane + kTmY + 128 * yb + 64 + 16 * b, ao);
        ok = ok && mbar_wait(&sc.solve_blk[b], (uint32_t)c & 1u);
        if (b > 0) {
          float r[16];
          horner16(base, kPbOff, yb, b, w, DBLK + yb * 256, trs, r);
#pragma unroll
          for (int t = 0; t < 16; ++t) ao[t] = fmaf(pc, ao[t], r[t]);
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) ao[t] *= pc;
        }
        float uu[16], gam[16];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 x = jt4(UB, j, 16 * b + 4 * q4);
          const float4 g = jt4(GAM, j, 16 * b + 4 * q4);
          uu[4 * q4] = x.x, uu[4 * q4 + 1] = x.y, uu[4 * q4 + 2] = x.z, uu[4 * q4 + 3] = x.w;
          gam[4 * q4] = g.x, gam[4 * q4 + 1] = g.y, gam[4 * q4 + 2] = g.z, gam[4 * q4 + 3] = g.w;
        }
        const float* pd = PD + b * 256;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float pcol[16];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const float4 x = *reinterpret_cast<const float4*>(pd + i * 16 + 4 * q4);
            pcol[4 * q4] = x.x, pcol[4 * q4 + 1] = x.y, pcol[4 * q4 + 2] = x.z,
                      pcol[4 * q4 + 3] = x.w;
          }
#pragma unroll
          for (int t = i; t < 16; ++t) ao[t] = fmaf(pcol[t], uu[i], gam[i] * ao[t]);
        }
        // o rows 16 b .. 16 b + 15 of column j into the swizzled o tile
#pragma unroll
        for (int t = 0; t < 16; ++t)
          *reinterpret_cast<__nv_bfloat16*>(ost + sw128_off(16 * b + t, j)) =
              __float2bfloat16_rn(ao[t]);
        pc *= DBLK[yb * 256 + b * 64 + j];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc.out_blk[b]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc.ybuf_free[yb]);
      fence_async_smem();
      if (named_sync_or(2, 64, !ok || *fail)) {
        *fail = 1;
        break;
      }
      if (tid == 64) {
        tma_store_3d(&tm_o, ost, 0, c * kF2C, (int)bh);
        bulk_commit();
      }
    }
    if (tid == 64) bulk_wait<0>();
  } else {
    // ======================= prep: one chunk ahead =======================
    const int p = tid - 128;  // row of [X; Q] (features), token / column half (scalars)
    const bool issuer = p == 0;
    auto load_chunk = [&](int cc) {
      const int sl = cc % kF2Ring;
      unsigned char* dst = base + kRingOff + sl * kSlot;
      mbar_expect_tx(&sc.full[sl], 3 * 8192);
      tma_load_3d(dst, &tm_k, 0, cc * kF2C - 1, (int)bh, &sc.full[sl]);
      tma_load_3d(dst + 8192, &tm_q, 0, cc * kF2C, (int)bh, &sc.full[sl]);
      tma_load_3d(dst + 16384, &tm_v, 0, cc * kF2C, (int)bh, &sc.full[sl]);
    };
    if (issuer)
      for (int cc = 0; cc < kF2Ring && cc < nch; ++cc) load_chunk(cc);
    const float eg = a.eps_gamma;
    for (int c = 0; c < nch; ++c) {
      const int slot = c % kF2Ring;
      const int64_t t0 = (int64_t)c * kF2C;
      const int n = (int)min((int64_t)kF2C, T - t0);
      unsigned char* xt = base + kRingOff + slot * kSlot;  // X, then Q at +8 KB
      unsigned char* vt = xt + 16384;
      bool ok = true;
      // gains of this thread's (token, column half), loaded early
      const int tt = p & 63, hh = p >> 6;
      float4 bet[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) bet[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (tt < n) {
        const float4* src =
            reinterpret_cast<const float4*>(a.beta + (rowbase + t0 + tt) * 64 + 32 * hh);
#pragma unroll
        for (int i = 0; i < 8; ++i) bet[i] = src[i];
      }
      const float lam_t = (p < 64 && p < n) ? a.lambda[rowbase + t0 + p] : 0.f;
      ok = ok && mbar_wait(&sc.full[slot], (uint32_t)(c / kF2Ring) & 1u);
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
      }
      // phi's scale of row p (p < 64: x_p = phi(k_{t0+p-1}); else phi(q_{t0+p-64}))
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
      const float nr = carried ? 1.f : phi_scale(ss, 64, a.phi);
      sc.nrm[p] = nr;
      if (p < 64) {
        const float E = ss * nr * nr;
        const float lam = ridge_of(lam_t, E, a.ridge);
        const float den = E + lam + a.eps;
        const bool sentinel = t0 + p == 0 && a.x_prev == nullptr;
        sc.E[p] = E;
        sc.lamr[p] = lam;
        sc.inv[p] = (!sentinel && p < n && den > 0.f) ? 1.f / den : 0.f;
      }
      // the Gram has read the raw rows: write phi's rows in place
      ok = ok && mbar_wait(&sc.gdone, (uint32_t)c & 1u);
      tc_fence_after();
      if (!carried) {
#pragma unroll
        for (int i = 0; i < 64; ++i) row[i] *= nr;
        put_row64(xt, p, row);
      }
      fence_async_smem();
      if (named_sync_or(3, 128, !ok || *fail)) {
        *fail = 1;
        break;
      }
      if (issuer) mbar_arrive(&sc.xq[slot]);
      // eta, gamma, eta v of token tt, columns 32 hh .. 32 hh + 31
      float ve[32], ge[32], ee[32];
      {
        float vv[32];
        load_half_sw(vt, tt, hh, vv);
        const float inv = sc.inv[tt], lam = sc.lamr[tt];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float bb[4] = {bet[i].x, bet[i].y, bet[i].z, bet[i].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float eta = bb[e] * inv;
            const float al = eta * lam;
            ee[4 * i + e] = eta;
            ge[4 * i + e] = al >= 1.f - eg ? eg : 1.f - al;
            ve[4 * i + e] = eta * vv[4 * i + e];
          }
        }
      }
      // the previous chunk's solve and output are done with these buffers
      if (c > 0) {
        ok = ok && mbar_wait(&sc.decu_done, (uint32_t)(c - 1) & 1u);
        ok = ok && mbar_wait(&sc.out_blk[3], (uint32_t)(c - 1) & 1u);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int jj = 32 * hh + i;
        ETA[jt(jj, tt)] = ee[i];
        GAM[jt(jj, tt)] = ge[i];
        ETAV[jt(jj, tt)] = ve[i];
      }
      // Gram readback: rows 0..63 K = X X^T (l < t), rows 64..127 P0 = Q X^T (l <= t)
      {
        float d[64];
        tmem_ld32(tlane + kTmG, d);
        tmem_ld32(tlane + kTmG + 32, d + 32);
        const bool krow = p < 64;
        const int t = p & 63, bt = t >> 4, tl = t & 15;
        float* dg = (krow ? KD : PD) + bt * 256;
#pragma unroll
        for (int l = 0; l < 64; ++l) {
          const bool keep = krow ? (l < t) : (l <= t);
          d[l] = keep ? d[l] * nr * sc.nrm[l] : 0.f;
        }
        put_row64(base + (krow ? kKbOff : kPbOff), t, d);
#pragma unroll
        for (int k = 0; k < 16; ++k) dg[k * 16 + tl] = d[16 * bt + k];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc.pre_ready);
      if (!ok) *fail = 1;
      // refill: chunk c + 2 into the slot of chunk c - 1 once its chain is done
      if (issuer && c >= 1 && c + 2 < nch) {
        const int sl = (c + 2) % kF2Ring;
        if (mbar_wait(&sc.empty[sl], (uint32_t)((c - 1) / kF2Ring) & 1u))
          load_chunk(c + 2);
        else
          *fail = 1;
      }
    }
    // x_last = phi(k_{T-1})
    if (a.x_last && warp == 4) {
      const __nv_bfloat16* kl = reinterpret_cast<const __nv_bfloat16*>(a.k) + (rowbase + T - 1) * 64;
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
  CUtensorMap tm_k, tm_q, tm_v, tm_o;
  if (!encode_rows_bf16(&tm_k, a.k, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kF2C) ||
      !encode_rows_bf16(&tm_q, a.q, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kF2C) ||
      !encode_rows_bf16(&tm_v, a.v, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kF2C) ||
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
  return cudaLaunchKernelEx(&cfg, tc_falcon2_chunk_kernel, a, nch, err, tm_k, tm_q, tm_v, tm_o);
}

}  // namespace falcon
