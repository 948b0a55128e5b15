// Building blocks shared by the tensor-core kernels (forward map kernel and
// the backward chunk kernel): bf16 packing, the 128-byte swizzled half-row
// accessors of 64-wide tiles, phi's scale, and the unit-lower inverse of a
// 64 x 64 chunk matrix (fp32 diagonal blocks, warp MMAs below them).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace falcon {
namespace tcu {
namespace {

using namespace tc;

// Chunk map of the m = d_v = 64 tensor-core forward, per (head, chunk): Mc as
// the scan's A operand, Nc, e^{g_C}.
constexpr uint32_t kMcBytes = 128 * 128;  // 128 rows x 64 bf16 (swizzled operand image)
constexpr uint32_t kNcBytes = 128 * 128;  // 128 rows x 64 bf16 (rows swizzled by 16 B)
constexpr uint32_t kMapBytes = kMcBytes + kNcBytes + 128;  // + e^{g_C} (padded)

// 1024-byte aligned base inside the dynamic shared buffer.  The offset is added
// to the __shared__ pointer itself (not via an integer round trip), so the
// compiler keeps the shared address space and emits shared loads and stores.
__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  const uint32_t off = (1024u - (smem_addr(p) & 1023u)) & 1023u;
  return p + off;
}

__device__ __forceinline__ void flag_error(int* err) {
  if (err) atomicExch(err, 1);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 8 consecutive values (scaled) as one 16-byte bf16 chunk.
__device__ __forceinline__ uint4 pack8(const float* v, float scale) {
  uint4 pk;
  pk.x = pack_bf16(scale * v[0], scale * v[1]);
  pk.y = pack_bf16(scale * v[2], scale * v[3]);
  pk.z = pack_bf16(scale * v[4], scale * v[5]);
  pk.w = pack_bf16(scale * v[6], scale * v[7]);
  return pk;
}

// Warp-level bf16 MMA, 16 x 8 x 16, fp32 accumulate (used for the 16-row
// blocks of the triangular solve, below the 64-row minimum of tcgen05).
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Half-row helpers: a thread owns columns 32h .. 32h+31 of row r (four
// 16-byte chunks) of a 64-wide bf16 tile with the 128-byte swizzle.
__device__ __forceinline__ void load_half_sw(const unsigned char* tile, int r, int h, float* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 pk =
        *reinterpret_cast<const uint4*>(tile + r * 128 + (((4 * h + c) ^ (r & 7)) << 4));
    const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&pk);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(hv[e]);
      v[8 * c + 2 * e] = f.x;
      v[8 * c + 2 * e + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void store_half_sw(unsigned char* tile, int r, int h, const float* v,
                                              float scale) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(tile + r * 128 + (((4 * h + c) ^ (r & 7)) << 4)) =
        pack8(v + 8 * c, scale);
}

// Scales, in place, the four chunks of the half row (one chunk at a time).
__device__ __forceinline__ void scale_half_sw(unsigned char* tile, int r, int h, float scale) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4* p = reinterpret_cast<uint4*>(tile + r * 128 + (((4 * h + c) ^ (r & 7)) << 4));
    const uint4 pk = *p;
    const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&pk);
    float v[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(hv[e]);
      v[2 * e] = f.x;
      v[2 * e + 1] = f.y;
    }
    *p = pack8(v, scale);
  }
}

__device__ __forceinline__ float sumsq32(const float* v) {
  float p[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 32; ++j) p[j & 7] += v[j] * v[j];
  return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}

// phi's scale for a row of m values with squared norm ss: 1 / max(||u||,
// 1e-12) for the l2 map (0 for an all-zero row, which makes no difference to
// phi(u) = 0 and keeps products with the exponential factors finite),
// 1 / sqrt(ss / m + eps_rms) for RMSNorm, 1 for the identity.
__device__ __forceinline__ float phi_scale(float ss, int m, int phi) {
  if (phi == FALCON_PHI_RMS) return rsqrtf(ss / (float)m + kEpsRms);
  if (phi != FALCON_PHI_L2) return 1.f;
  return ss > 0.f ? rsqrtf(fmaxf(ss, 1e-24f)) : 0.f;
}

// ---- T = (I + A)^{-1} for a 64 x 64 chunk, off-diagonal blocks in registers ----
// Byte offset of 16-byte chunk c of row r in a 64-wide bf16 tile with the
// 128-byte swizzle.
__device__ __forceinline__ uint32_t sw_chunk(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// Four 8 x 8 bf16 matrices from shared memory in the mma.sync A-fragment
// layout (lanes 0-7, 8-15, 16-23, 24-31 give the row addresses of matrices
// 0..3).
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr)
               : "memory");
}

// Two 8 x 8 bf16 matrices, transposed on the way (rows of a row-major K x N
// tile become the mma.sync B fragment; lanes 0-15 give the row addresses).
__device__ __forceinline__ void ldsm_x2_trans(uint32_t (&r)[2], uint32_t saddr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(saddr)
               : "memory");
}

// Transpose of an 8 x 8 bf16 matrix held one 32-bit pair per lane (row
// lane / 4, columns 2 (lane % 4) and +1) across the warp.
__device__ __forceinline__ uint32_t movm_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

constexpr int kLdD = 17;  // fp32 row stride of the diagonal blocks of A

// Byte offset of 16-byte chunk c (0 or 1) of row r in the copy of T's
// diagonal blocks (32-byte rows, the chunk flipped every four rows so that
// ldmatrix row reads do not collide in shared-memory banks).
__device__ __forceinline__ uint32_t dblk_chunk(int r, int c) {
  return (uint32_t)(r * 32 + ((c ^ ((r >> 2) & 1)) << 4));
}

// T = (I + A)^{-1} for the strictly lower 64 x 64 A, eight warps.  The result
// leaves with its columns scaled, T Diag(col_scale), as bf16 in the 128-byte
// swizzled 64 x 64 tile t_tile (rows, the K-major operand image), zero above
// the diagonal blocks.  Inputs: a_tile, A as bf16 in the same layout; a_diag,
// the fp32 diagonal blocks (row i holds A[i][16 (i / 16) + k], k = 0..15, rows
// of kLdD floats); col_scale, 64 floats (kScaled; otherwise T itself is
// stored).  d_blk (2 KB) receives the unscaled diagonal blocks of T as bf16,
// which the strips below read.
//
// Diagonal block b is inverted in fp32 by forward substitution, one thread
// per column (threads 0..63: block tid / 16, column tid % 16): going down the
// column, t_i = delta_ij - sum_{k<i} A_ik t_k with the fused multiply-adds in
// the order k = 0, 1, ..., the rows of A broadcast from shared memory; the
// other warps have no part in it.
// Below it,
// T_{b,<b} = T_bb (-A_{b,<b} T_{<b}) splits into independent 8-column strips:
// strip n (columns 8n .. 8n+7, n = 0..5) of block row b needs only strip n of
// the block rows above it.  Warp n runs its
// strip down the block rows with warp MMAs, keeping each finished block as
// the next MMA's B operand in registers: an accumulator tile, packed to bf16,
// is transposed across the warp by movmatrix into operand layout, so neither
// the right-hand side nor the finished blocks go through shared memory and the
// warps do not wait on one another.  The MMA operands (A, the diagonal
// blocks, the right-hand sides and the finished blocks) are bf16, the
// accumulation fp32; the column scaling enters only the stored copy.  The
// caller fences and synchronises before t_tile is read.
template <bool kScaled>
__device__ void solve_unit_lower_sw(const unsigned char* a_tile, const float* a_diag,
                                    unsigned char* t_tile, unsigned char* d_blk,
                                    const float* col_scale) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < 64) {
    const int b = tid >> 4, j = tid & 15;
    const float* L = a_diag + 16 * b * kLdD;
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = (i == j) ? 1.f : 0.f;
#pragma unroll
      for (int k = 0; k < i; ++k) acc = fmaf(-L[i * kLdD + k], t[k], acc);
      t[i] = acc;
    }
    // Column j of T_bb: unscaled into d_blk, scaled into t_tile; each thread
    // also zeroes the chunks of row 16 b + j right of the diagonal block.
    const float cs = kScaled ? col_scale[16 * b + j] : 1.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int row = 16 * b + i;
      *reinterpret_cast<__nv_bfloat16*>(d_blk + dblk_chunk(row, j >> 3) + 2 * (j & 7)) =
          __float2bfloat16_rn(t[i]);
      *reinterpret_cast<__nv_bfloat16*>(t_tile + sw_chunk(row, 2 * b + (j >> 3)) +
                                        2 * (j & 7)) = __float2bfloat16_rn(t[i] * cs);
    }
    for (int z = 2 * b + 2; z < 8; ++z)
      *reinterpret_cast<uint4*>(t_tile + sw_chunk(16 * b + j, z)) = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();  // diagonal blocks of T complete
  if (warp < 6) {
    const int nt = warp, kb0 = nt >> 1, g = lane >> 2, t = lane & 3;
    const int la = (lane & 7) + 8 * ((lane >> 3) & 1), ca = lane >> 4;
    const uint32_t abase = smem_addr(a_tile), dbase = smem_addr(d_blk);
    const float cs0 = kScaled ? col_scale[8 * nt + 2 * t] : 1.f;
    const float cs1 = kScaled ? col_scale[8 * nt + 2 * t + 1] : 1.f;
    uint32_t tb[4][2];  // finished blocks (kb, strip) as B fragments, unscaled
#pragma unroll
    for (int kb = 0; kb < 3; ++kb)
      if (kb == kb0) ldsm_x2_trans(tb[kb], dbase + dblk_chunk(16 * kb + la, nt & 1));
#pragma unroll
    for (int b = 1; b < 4; ++b) {
      if (b <= kb0) continue;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kb = 0; kb < b; ++kb) {
        if (kb < kb0) continue;
        uint32_t fa[4];
        ldsm_x4(fa, abase + sw_chunk(16 * b + la, 2 * kb + ca));
        mma16816(acc, fa, tb[kb]);
      }
      // R = -A_{b,<b} T_{<b} (strip nt) as the B operand of T_bb R.
      const uint32_t rb[2] = {movm_trans(pack_bf16(-acc[0], -acc[1])),
                              movm_trans(pack_bf16(-acc[2], -acc[3]))};
      uint32_t fd[4];
      ldsm_x4(fd, dbase + dblk_chunk(16 * b + la, ca));
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      mma16816(c, fd, rb);
      const int r0 = 16 * b + g;
      *reinterpret_cast<uint32_t*>(t_tile + sw_chunk(r0, nt) + 4 * t) =
          pack_bf16(c[0] * cs0, c[1] * cs1);
      *reinterpret_cast<uint32_t*>(t_tile + sw_chunk(r0 + 8, nt) + 4 * t) =
          pack_bf16(c[2] * cs0, c[3] * cs1);
      if (b < 3) {
        tb[b][0] = movm_trans(pack_bf16(c[0], c[1]));
        tb[b][1] = movm_trans(pack_bf16(c[2], c[3]));
      }
    }
  }
}

}  // namespace
}  // namespace tcu
}  // namespace falcon
