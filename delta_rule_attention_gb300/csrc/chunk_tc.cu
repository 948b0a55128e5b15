// Tensor-core (tcgen05) chunked forward for bf16 inputs with m = d_v in
// {64, 128} and chunk C = 64.
//
// Two launches:
//
//  1. tc_chunk_map_kernel<M> -- all chunks in parallel (one CTA per chunk for
//     m = 64, two for m = 128, each taking one column half).  It turns the
//     chunk into an affine map of the state entering it (the chunk-local
//     log-space form of the positive-decay renormalisation of page
//     hyper.ai/fr/papers/2608.27763, Section 4.4 Eq. (4.15)-(4.16); WY/UT form
//     with one triangular solve per chunk, as the complexity table of page
//     juhoplayground.github.io describes):
//
//        S'  = e^{g_C} S + Mc_top S + Nc_top,   Mc_top = -Xt^T W,    Nc_top = Xt^T U~
//        O   =             Mc_bot S + Nc_bot,   Mc_bot = Diag(e^g) Q - P W,  Nc_bot = P U~
//
//     with W = T Diag(eta e^{g_-}) X, U~ = T Diag(eta) V, T = (I + A)^{-1}.
//     tcgen05 MMAs (bf16 operands in shared memory, fp32 accumulators in TMEM)
//     do the contractions:
//        MMA1   [K; Q] K^T (raw rows)      -> Gram of the write features, Q X^T
//        MMA2   [Xh^T; Vh^T] T^T           -> [W^T; U~^T]
//        MMA3   [Xt^T; P] [W | U~]         -> [Xt^T W | Xt^T U~ ; P W | P U~]
//     The unit-lower solve runs in fp32 on the diagonal 16 x 16 blocks; the
//     blocks below them follow in 8-column strips, one warp each, with warp
//     MMAs whose operands stay in registers.  The map goes to the workspace
//     as ready-to-use bf16 tiles (Mc swizzled as an MMA operand, Nc with rows
//     swizzled at 16-byte granularity) plus e^{g_C}.
//     Falcon-1A takes the same path with T = I and W = 0.
//
//  2. tc_chunk_scan_kernel (m = 64) / tc_chunk_scan128_kernel (m = 128) --
//     sequential over chunks, one CTA per head (per head and d_v slice for
//     m = 128): per chunk the state MMA [Mc_top; Mc_bot] S, with the maps of
//     the next chunks prefetched.  The e^{g_C} S part of the state update
//     stays in fp32 registers (only the correction goes through bf16
//     operands), so an undecayed state does not drift over long sequences.
#include <cuda_bf16.h>

#include <atomic>
#include <type_traits>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tc_util.cuh"
#include "tmap.cuh"

namespace falcon {

namespace {

using namespace tc;
using namespace tcu;

constexpr int kC = 64;
constexpr int kScanRing = 5;  // map stages the m = 64 scan loads before its first MMA
// A chunk whose log-decay spans at most this much factors e^{a-b} as
// e^{a-r} e^{r-b} (both factors stay within fp32 range).
constexpr float kFactorSpan = 80.f;

// ---------------------------------------------------------------------------
// Map kernel.  One CTA per (head, chunk) for m = d_v = 64; for m = d_v = 128
// two CTAs per chunk, CTA j taking the column half j of W, U~ and of the map
// (K-atom j of Mc, d_v slice j of Nc); the Gram matrix, the solve and T are
// the same in both.  Shared memory, in bytes from a 1024-aligned base (buffers
// with disjoint lifetimes share space), m = 64 (52 KB, four CTAs per SM):
//   K   [0, 8192)       raw k rows t0-1 .. t0+62 as landed by TMA (128B-swizzled;
//                       row r holds the write feature x_r before phi) -> Xh
//                       (MMA2's A, atom 0) -> Xt (atom 0 of MMA3a's MN-major A)
//   Q   [8192, 16384)   raw q rows as landed by TMA; [K; Q] is MMA1's A operand
//                       -> AD, the fp32 diagonal 16 x 16 blocks of A (rows of
//                       17), and DB at 12544, the unscaled diagonal blocks of T
//                       -> zero tile (atom 1 of MMA3a; rows 0..63 of MMA3b)
//   P   [16384, 24576)  P (rows 64..127 of MMA3b, K-major)
//   A   [24576, 32768)  A as bf16 (the solve's MMA operand)  } [W^T; U~^T] (MMA3's
//   T   [32768, 40960)  T = (I + A)^{-1} as bf16 (MMA2's B) } B) -> Nc staging
//   VH  [40960, 49152)  raw v rows as landed by TMA (atom 1 of MMA2's A)
//   SC  [49152, ...)    per-token scalars and barriers
// m = 128 (68 KB, three CTAs per SM): [K; Q] is two K-atoms of 16 KB,
// [K_a0 | Q_a0 | K_a1 | Q_a1] (columns 0..63 and 64..127); afterwards Xt's
// two M-atoms replace K_a0 and K_a1, P replaces Q_a0, and the dead q rows of
// Q_a1 take AD and DB.  A, T, XH, VH and SC follow at 32768, 40960, 49152,
// 57344 and 65536 (XH holds the x columns and VH the v columns of half j).
// MMA3 runs in two passes through the same 128 TMEM columns: the output rows
// ([junk; P] [W | U~]) first, staged over the dead XH and VH tiles, then the
// state rows (Xt^T [W | U~]), staged over the first 16 KB (Xt's first atom
// and P) and over [W^T; U~^T].
// T carries the step sizes in its columns, T' = T Diag(eta), so that
// MMA2 = [Xh^T; V^T] T'^T gives W^T = (T Diag(eta e^{g_-}) X)^T with
// Xh = Diag(e^{g_-}) X and U~^T = (T Diag(eta) V)^T from the raw v rows.
// MMA1 runs on the raw bf16 rows; phi's normalisation enters afterwards as
// fp32 row and column scalings of the accumulators and of the later operand
// copies.
template <int M>
struct MapLayout;
// m = 64 (four CTAs per SM): buffers are reused as their contents die:
//   K   raw k rows -> Xh (once MMA1 has read K) -> Xt (once MMA2 has read Xh)
//       -> with Q, the Mc staging;
//   Q   raw q rows -> the fp32 diagonal blocks of A (AD) and the solve's bf16
//       diagonal blocks of T (DB), once MMA1 has read Q -> the zero tile of
//       MMA3 (once the solve is done);
//   A and T, contiguous: A and T -> [W^T; U~^T] (MMA3's B) -> the Nc staging.
template <>
struct MapLayout<64> {
  static constexpr uint32_t K = 0, Q = 8192, P = 16384, A = 24576, T = 32768, VH = 40960,
                            SC = 49152;
  static constexpr uint32_t XH = K, AD = Q, DB = Q + 4352;
  static constexpr uint32_t kAtom = 0;  // K-atom stride of [K; Q] (one atom)
  static constexpr int kHalves = 1;
  static constexpr int kMinBlocks = 4;
  static constexpr uint32_t kTmemCols = 128;
  static constexpr uint32_t kMapBytes = 128 * 128 * 2 + 128;  // Mc, Nc, e^{g_C}
};
// m = 128 (three CTAs per SM): the q rows of the second K-atom are dead once
// MMA1 has read them and take the solve's diagonal blocks (AD, DB).
template <>
struct MapLayout<128> {
  static constexpr uint32_t K = 0, Q = 8192, P = 8192, A = 32768, T = 40960, XH = 49152,
                            VH = 57344, SC = 65536;
  static constexpr uint32_t AD = Q + 16384, DB = AD + 4352;
  static constexpr uint32_t kAtom = 16384;
  static constexpr int kHalves = 2;
  static constexpr int kMinBlocks = 3;
  static constexpr uint32_t kTmemCols = 128;
  // Per chunk: Mc K-atoms 0 and 1 (192 rows x 128 B each: 128 state rows,
  // then 64 output rows), Nc d_v slices 0 and 1 (192 rows x 128 B), e^{g_C}.
  static constexpr uint32_t kMcAtom = 192 * 128;
  static constexpr uint32_t kMapBytes = 4 * kMcAtom + 128;
};
constexpr bool map_layout128_ok() {
  using L = MapLayout<128>;
  return L::A % 1024 == 0 && L::T == L::A + 8192 && L::XH % 1024 == 0 &&
         L::XH >= L::T + 8192 && L::VH == L::XH + 8192 && L::SC >= L::VH + 8192 &&
         L::AD == L::Q + L::kAtom && L::AD + 64 * kLdD * 4 <= L::DB && L::DB % 16 == 0 &&
         L::DB + 2048 <= L::AD + 8192 && L::SC % 16 == 0;
}
constexpr bool map_layout64_ok() {
  using L = MapLayout<64>;
  return L::K % 1024 == 0 && L::Q == L::K + 8192 && L::P == L::Q + 8192 && L::A % 1024 == 0 &&
         L::T == L::A + 8192 && L::VH % 1024 == 0 && L::VH >= L::T + 8192 &&
         L::AD + 64 * kLdD * 4 <= L::DB && L::DB % 16 == 0 && L::DB + 2048 <= L::Q + 8192 &&
         L::SC >= L::VH + 8192 && L::SC % 16 == 0;
}
static_assert(map_layout64_ok() && map_layout128_ok(), "map kernel shared-memory layout");

// A thread's raw half row (32 bf16 input values) kept as 16 packed bf16
// pairs: exact, half the registers of fp32.
__device__ __forceinline__ float bf16_at(const uint32_t (&p)[16], int i) {
  return __uint_as_float((i & 1) ? (p[i >> 1] & 0xffff0000u) : (p[i >> 1] << 16));
}
__device__ __forceinline__ void load_half_raw(const unsigned char* tile, int r, int h,
                                              uint32_t (&p)[16]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 pk =
        *reinterpret_cast<const uint4*>(tile + r * 128 + (((4 * h + c) ^ (r & 7)) << 4));
    p[4 * c] = pk.x;
    p[4 * c + 1] = pk.y;
    p[4 * c + 2] = pk.z;
    p[4 * c + 3] = pk.w;
  }
}
__device__ __forceinline__ float sumsq_packed(const uint32_t (&p)[16]) {
  float q[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 32; ++i) q[i & 7] = fmaf(bf16_at(p, i), bf16_at(p, i), q[i & 7]);
  return ((q[0] + q[1]) + (q[2] + q[3])) + ((q[4] + q[5]) + (q[6] + q[7]));
}
// The half row times `scale`, as bf16, into a 128B-swizzled tile row.
__device__ __forceinline__ void store_half_packed(unsigned char* tile, int r, int h,
                                                  const uint32_t (&p)[16], float scale) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = bf16_at(p, 8 * c + e);
    *reinterpret_cast<uint4*>(tile + r * 128 + (((4 * h + c) ^ (r & 7)) << 4)) = pack8(v, scale);
  }
}

// A thread's raw half row: packed bf16 pairs where registers are short (m = 64,
// four CTAs per SM), fp32 otherwise; the same values and products either way.
template <bool kPacked>
struct HalfRow;
template <>
struct HalfRow<true> {
  uint32_t p[16];
  __device__ __forceinline__ void load(const unsigned char* tile, int r, int h) {
    load_half_raw(tile, r, h, p);
  }
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < 16; ++i) p[i] = 0u;
  }
  __device__ __forceinline__ float at(int i) const { return bf16_at(p, i); }
  __device__ __forceinline__ float sumsq() const { return sumsq_packed(p); }
  __device__ __forceinline__ void store(unsigned char* tile, int r, int h, float scale) const {
    store_half_packed(tile, r, h, p, scale);
  }
};
template <>
struct HalfRow<false> {
  float v[32];
  __device__ __forceinline__ void load(const unsigned char* tile, int r, int h) {
    load_half_sw(tile, r, h, v);
  }
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
  }
  __device__ __forceinline__ float at(int i) const { return v[i]; }
  __device__ __forceinline__ float sumsq() const { return sumsq32(v); }
  __device__ __forceinline__ void store(unsigned char* tile, int r, int h, float scale) const {
    store_half_sw(tile, r, h, v, scale);
  }
};

struct MapScalars {
  float eta[64], g[64], gx[64];
  // Rank-1 decay factors (span <= kFactorSpan), with phi's scale of x_l in the
  // column factor: cu_l = e^{rr - g_l} / ||x_l||, fv_j = eta_j e^{g_{j-1} - rr},
  // fw_i = e^{g_i - rr}.
  float cu[64], fv[64], fw[64];
  float nrm[128];                // phi's scale of row r of [K; Q] (1 / ||row||, or 1)
  float ssp[2][128];             // half-row partial sums of squares
  int fail;
  uint64_t bar_in, bar_mma;
  uint32_t tmem_base;
};
template <int M>
constexpr size_t map_smem_bytes() {
  return MapLayout<M>::SC + sizeof(MapScalars);
}
constexpr int kMapThreads = 256;

// 256 threads per CTA: thread t owns row r = t & 127 (its TMEM lane) and
// columns 32h .. 32h+31 (h = t >> 7) of the CTA's 64-column half j.
// kNorm (m = 64, Falcon-1A): the launch also writes the normalised read's
// per-chunk terms to a.norm_ws (NormLayout): e^{g_t}, e^{g_C}, phi's scale of
// q_t, the increment y_C = sum_j eta_j e^{g_C - g_j} x_j (fp32, from the raw
// rows) and the in-chunk read r_t = sum_{j <= t} P_tj eta_j.  Falcon-1A has
// W = 0, so MMA3's W columns carry no map: column 0 of W is set to eta, and
// MMA3 returns r_t in column 0 of the output rows (the bf16 P and eta operands
// of the numerator's own in-chunk term P Diag(eta) V); the Mc staging zeroes
// that column again.
template <int M, bool kNorm = false>
__global__ void __launch_bounds__(kMapThreads, MapLayout<M>::kMinBlocks)
    tc_chunk_map_kernel(ChunkArgs a, int nchunks, int c_begin, int* err, uint32_t pf_ahead,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_v) {
  using L = MapLayout<M>;
  constexpr bool kWide = M == 128;
  static_assert(!kNorm || M == 64, "the normalised read's terms: m = 64");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* const base = align1024(smem_raw);
  unsigned char* const kt = base + L::K;
  unsigned char* const qt = base + L::Q;
  unsigned char* const p_tile = base + L::P;
  unsigned char* const a_tile = base + L::A;
  unsigned char* const t_tile = base + L::T;
  unsigned char* const xh_tile = base + L::XH;
  unsigned char* const wu_tile = base + L::A;  // [W^T; U~^T], later the Nc staging
  unsigned char* const vh = base + L::VH;
  MapScalars& sc = *reinterpret_cast<MapScalars*>(base + L::SC);
  float* const a_diag = reinterpret_cast<float*>(base + L::AD);
  unsigned char* const xt_tile = kt;    // MN-major A of MMA3a, atom 0
  unsigned char* const zero_tile = qt;  // m = 64: atom 1 of MMA3a; rows 0..63 of MMA3b

  const int c = c_begin + (int)(blockIdx.x / L::kHalves);
  const int j = blockIdx.x % L::kHalves;  // column half of this CTA
  const int64_t bh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = tid & 127, h = tid >> 7;
  const int64_t t0 = (int64_t)c * kC;
  const int n = (int)min((int64_t)kC, a.T - t0);
  const bool f1 = a.rule == kFalcon1;
  const bool last = c == nchunks - 1;
  const int64_t rowbase = bh * a.T;
  // Row 0 of the first chunk is x_1: x_prev as given (already phi-mapped), or
  // the sentinel zero (the TMA box starts at row -1, which reads as zeros).
  const bool carried_row = c == 0 && r == 0;
  const bool patch = c == 0 && a.x_prev != nullptr;
  const NormLayout nl{a.BH * nchunks, 64, kC};
  const size_t mi = (size_t)(bh * nchunks + c);
  float ypart = 0.f;  // kNorm: this lane's column of the increment over its warp's rows

  // Waits: with four CTAs per SM (m = 64) the other CTAs' phases run while one
  // waits, so it polls with a sleep between polls.
  auto wait = [](uint64_t* bar, uint32_t parity) {
    return M == 64 ? mbar_wait_backoff(bar, parity) : mbar_wait(bar, parity);
  };
  // TMEM is allocated by warp 1, so that thread 0 issues the input tile copies
  // (the head of the CTA's chain) without waiting for the allocation.
  if (warp == 1) tmem_alloc(&sc.tmem_base, L::kTmemCols);
  // Launched behind the previous call's scan (programmatic dependent launch),
  // the CTA may start while that grid still runs: no input is read, and no
  // output or workspace byte written, before the preceding grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    mbar_init(&sc.bar_in, 1);
    mbar_init(&sc.bar_mma, 1);
    fence_mbar_init();
    sc.fail = 0;
    // k rows t0-1 .. t0+62, q and v rows t0 .. t0+63 (rows past T read as zeros).
    mbar_expect_tx(&sc.bar_in, (kWide ? 5 : 3) * 8192);
    if constexpr (!kWide) {
      // The inputs are read once; the chunk maps this grid writes (101 MB on
      // the lm shape) are read again by the scan: the inputs leave L2 first.
      const uint64_t pol = l2_evict_first();
      tma_load_3d_hint(kt, &tm_k, 0, (int)(t0 - 1), (int)bh, &sc.bar_in, pol);
      tma_load_3d_hint(qt, &tm_q, 0, (int)t0, (int)bh, &sc.bar_in, pol);
      tma_load_3d_hint(vh, &tm_v, 64 * j, (int)t0, (int)bh, &sc.bar_in, pol);
    } else {
#pragma unroll
      for (int at = 0; at < (kWide ? 2 : 1); ++at) {
        tma_load_3d(kt + at * L::kAtom, &tm_k, 64 * at, (int)(t0 - 1), (int)bh, &sc.bar_in);
        tma_load_3d(qt + at * L::kAtom, &tm_q, 64 * at, (int)t0, (int)bh, &sc.bar_in);
      }
      tma_load_3d(vh, &tm_v, 64 * j, (int)t0, (int)bh, &sc.bar_in);
    }
  }
  // CTAs are dispatched close to linear block order, so the one that takes
  // this CTA's slot is about pf_ahead (the resident CTAs of the device) blocks
  // on: bring its k, q, v rows into L2 now, so that its tile loads hit L2.
  if (tid == 64 && pf_ahead > 0) {
    const uint32_t Lp = blockIdx.x + gridDim.x * blockIdx.y + pf_ahead;
    if (Lp < gridDim.x * gridDim.y) {
      const int cp = c_begin + (int)((Lp % gridDim.x) / L::kHalves);
      const int64_t rp = (int64_t)(Lp / gridDim.x) * a.T + (int64_t)cp * kC;  // first row
      const uint32_t bytes = (uint32_t)min((int64_t)kC, a.T - (int64_t)cp * kC) * M * 2;
      bulk_prefetch_l2(reinterpret_cast<const __nv_bfloat16*>(a.k) + rp * M, bytes);
      bulk_prefetch_l2(reinterpret_cast<const __nv_bfloat16*>(a.q) + rp * M, bytes);
      bulk_prefetch_l2(reinterpret_cast<const __nv_bfloat16*>(a.v) + rp * M, bytes);
    }
  }
  // Warps 0 and 1 form the step sizes of all 64 tokens (lane l: tokens l and
  // l + 32), so each has the whole prefix without an exchange.
  // The scan opens with the first kScanRing maps of every head, most of them
  // written early in this grid and out of L2 by its end: the last resident set
  // of CTAs brings them back (CTA k of that set: head k % BH, chunk k / BH).
  if constexpr (M == 64) {
    if (tid == 96 && pf_ahead > 0 && c_begin == 0) {
      const uint32_t total = gridDim.x * gridDim.y;
      const uint32_t Lc = blockIdx.x + gridDim.x * blockIdx.y;
      if (Lc + pf_ahead >= total) {
        const uint32_t k = Lc + pf_ahead - total;
        const uint32_t hh = k % gridDim.y, cc = k / gridDim.y;
        if (cc < (uint32_t)kScanRing && (int)cc < nchunks)
          bulk_prefetch_l2(reinterpret_cast<const unsigned char*>(a.workspace) +
                               ((size_t)hh * nchunks + cc) * L::kMapBytes,
                           L::kMapBytes);
      }
    }
  }
  float beta2[2] = {0.f, 0.f}, lam2[2] = {0.f, 0.f};
  if (warp < 2) {
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      if (lane + 32 * k2 < n) {
        beta2[k2] = a.beta[rowbase + t0 + lane + 32 * k2];
        lam2[k2] = a.lambda[rowbase + t0 + lane + 32 * k2];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sc.tmem_base;
  const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  if (!wait(&sc.bar_in, 0)) sc.fail = 1;
  if (patch) {
    // x_1 = x_prev in row 0 of the K tile (bf16) for MMA1.
    if (tid < 8 * (M / 64)) {
      const int at = tid >> 3, ch = tid & 7;
      float v8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v8[e] = a.x_prev[bh * M + 64 * at + 8 * ch + e];
      // row 0: no swizzle shift
      *reinterpret_cast<uint4*>(kt + at * L::kAtom + (ch << 4)) = pack8(v8, 1.f);
    }
    fence_async_smem();
    __syncthreads();
  }

  // ---- MMA1: D[0:64) = [K; Q] K^T on the raw rows, issued before the features ----
  if (tid == 0 && !sc.fail) {
    tc_fence_after();
#pragma unroll
    for (int at = 0; at < (kWide ? 2 : 1); ++at)
      mma_k64(tmem, smem_addr(kt + at * L::kAtom), false, 16, smem_addr(kt + at * L::kAtom),
              false, 16, idesc_bf16(128, 64, false, false), at > 0);
    mma_commit(&sc.bar_mma);
  }

  // ---- features: rows 0..63 are the write features x_r = phi(k_{t0+r-1}),
  //      rows 64..127 are phi(q_{t0+r-64}); a thread keeps its raw half row
  //      (of column half j) and the row's phi scale nr.  m = 128: the other
  //      half (xo) enters the norm and Xt.
  // The raw half rows (xp: half j, xo: the other half, m = 128); the carried
  // row (x_prev, fp32) is read again from global memory where it is used.
  const bool carried_fp32 = carried_row && a.x_prev != nullptr;
  HalfRow<true> xp, xo;
  if (carried_fp32) {
    float x[32], y[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = a.x_prev[bh * M + 64 * j + 32 * h + i];
    if (kWide) {
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = a.x_prev[bh * M + 64 * (1 - j) + 32 * h + i];
    }
    if (kWide)  // same summation order in both halves' CTAs
      sc.ssp[h][r] = j == 0 ? sumsq32(x) + sumsq32(y) : sumsq32(y) + sumsq32(x);
    else
      sc.ssp[h][r] = sumsq32(x);
    xp.clear();  // not used for this row
    xo.clear();
  } else {
    const unsigned char* rt = (r < 64 ? kt : qt);
    xp.load(rt + j * L::kAtom, r & 63, h);
    if (kWide) xo.load(rt + (1 - j) * L::kAtom, r & 63, h);
    if (kWide)
      sc.ssp[h][r] = j == 0 ? xp.sumsq() + xo.sumsq() : xo.sumsq() + xp.sumsq();
    else
      sc.ssp[h][r] = xp.sumsq();
  }
  // This thread's half row (half `part`: j or the other) times `scale` into a tile row.
  auto store_row = [&](unsigned char* tile, int row, int part, float scale) {
    if (carried_fp32) {
      float v[32];
      const int jj = part == 0 ? j : 1 - j;
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = a.x_prev[bh * M + 64 * jj + 32 * h + i];
      store_half_sw(tile, row, h, v, scale);
    } else {
      (part == 0 ? xp : xo).store(tile, row, h, scale);
    }
  };
  __syncthreads();
  const float ss = sc.ssp[0][r] + sc.ssp[1][r];
  const float nr = carried_row ? 1.f : phi_scale(ss, M, a.phi);
  if (h == 0) sc.nrm[r] = nr;
  if constexpr (kNorm) {
    if (h == 0 && r >= 64) a.norm_ws[nl.nq() + mi * kC + (r - 64)] = r - 64 < n ? nr : 1.f;
  }
  if (a.x_last && last) {
    // phi(k_{T-1}) (columns of half j): row n of the features when the last
    // chunk is partial, otherwise the row after the K tile, from global memory.
    float* xl = a.x_last + bh * M + 64 * j + 32 * h;
    if (n < kC && r == n) {
#pragma unroll
      for (int i = 0; i < 32; ++i) xl[i] = xp.at(i) * nr;
    } else if (n == kC && r == 64) {
      const __nv_bfloat16* kl =
          reinterpret_cast<const __nv_bfloat16*>(a.k) + (rowbase + a.T - 1) * M;
      float part[32];
      float s2 = 0.f;
      for (int pc = 0; pc < M / 32; ++pc) {  // fixed order over the whole row
#pragma unroll
        for (int i = 0; i < 32; ++i) part[i] = __bfloat162float(kl[32 * pc + i]);
        s2 += sumsq32(part);
      }
      const float s = phi_scale(s2, M, a.phi);
#pragma unroll
      for (int i = 0; i < 32; ++i) xl[i] = __bfloat162float(kl[64 * j + 32 * h + i]) * s;
    }
  }

  // ---- step sizes, log-decays, chunk-local inclusive prefix g and the rank-1
  //      decay factors (warps 0 and 1; thread t < 64 publishes token t's) ----
  if (warp < 2) {
    float etav[2], lgv[2];
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int tk = lane + 32 * k2;  // token t0 + tk, write-feature row tk
      const float ssk = sc.ssp[0][tk] + sc.ssp[1][tk];
      const float nrk = (c == 0 && tk == 0) ? 1.f : phi_scale(ssk, M, a.phi);
      const float Ek = ssk * nrk * nrk;  // ||x_tk||^2
      etav[k2] = 0.f;
      lgv[k2] = 0.f;
      if (tk < n) {
        float gam;
        const bool sentinel = (t0 + tk == 0) && (a.x_prev == nullptr);
        etav[k2] = step_eta_gamma(sentinel, Ek, beta2[k2], ridge_of(lam2[k2], Ek, a.ridge),
                                  a.eps, a.eps_gamma, &gam, &lgv[k2]);
      }
    }
    float incl[2] = {lgv[0], lgv[1]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const float y = __shfl_up_sync(0xffffffffu, incl[k2], o);
        if (lane >= o) incl[k2] += y;
      }
    }
    incl[1] += __shfl_sync(0xffffffffu, incl[0], 31);
    const float gCw = __shfl_sync(0xffffffffu, incl[1], 31);
    const float eo = warp == 0 ? etav[0] : etav[1];  // this thread's token, t = tid
    const float lo = warp == 0 ? lgv[0] : lgv[1];
    const float go = warp == 0 ? incl[0] : incl[1];
    sc.eta[tid] = eo;
    sc.g[tid] = go;
    sc.gx[tid] = go - lo;
    if constexpr (kNorm) {
      a.norm_ws[nl.eg() + mi * kC + tid] = __expf(go);
      if (tid == 0) a.norm_ws[nl.dec() + mi * 4] = __expf(gCw);
    }
    // Rank-1 decay factors around rr = g_C / 2: e^{rr - g_l} (times phi's scale
    // of x_l), fv_j = eta_j e^{g_{j-1} - rr}, fw_i = e^{g_i - rr}.
    if (-gCw <= kFactorSpan) {
      const float rr = 0.5f * gCw;
      sc.cu[tid] = __expf(rr - go) * nr;
      sc.fv[tid] = eo * __expf((go - lo) - rr);
      sc.fw[tid] = __expf(go - rr);
    }
  }
  __syncthreads();  // step sizes, prefix and decay factors visible
  const float gC = sc.g[kC - 1];
  const bool factored = -gC <= kFactorSpan;
  // Xh = Diag(e^{g_-}) X (MMA2's A, columns of half j; Falcon-1A: W = 0, so
  // Xh = 0): m = 128 into its own tile now; m = 64 into the K tile once MMA1
  // has read it.
  const float xh_scale = f1 ? __expf(sc.gx[r & 63]) * nr : 0.f;
  if (r < 64) {
    if (kWide) store_row(xh_tile, r, 0, xh_scale);
    // Falcon-1A: T' = Diag(eta), whose rows are written here (the solve writes
    // Falcon-1's).
    if (!f1) {
      float trow[32];
      const float er = sc.eta[r];
#pragma unroll
      for (int i = 0; i < 32; ++i) trow[i] = (32 * h + i == r) ? er : 0.f;
      store_half_sw(t_tile, r, h, trow, 1.f);
    }
  }
  // Every thread sees MMA1 complete before it overwrites the K and Q tiles.
  if (!sc.fail && !wait(&sc.bar_mma, 0)) sc.fail = 1;
  tc_fence_after();
  if (!kWide) {
    if (r < 64) store_row(xh_tile, r, 0, xh_scale);
  } else if (r < 64) {
    // Xt = Diag(e^{g_C - g}) X over the K atoms (m = 128; m = 64 writes Xt
    // over Xh once MMA2 has read it)
    const float xs = __expf(gC - sc.g[r]) * nr;
    store_row(xt_tile + j * L::kAtom, r, 0, xs);
    store_row(xt_tile + (1 - j) * L::kAtom, r, 1, xs);
  }
  {
    // This warp's half rows may lie wholly above the diagonal (columns 32..63
    // of rows 0..31, warp-uniform): A there is never read by the solve and P
    // there is zero, so the warp skips the accumulator.
    const bool above = h == 1 && (warp & 1) == 0;
    if (r >= 64 && above) {
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        *reinterpret_cast<uint4*>(p_tile + sw_chunk(r - 64, 4 * h + cc)) =
            make_uint4(0u, 0u, 0u, 0u);
    } else if (!above && (r >= 64 || f1)) {
      float d[32];
      tmem_ld32(tlane + 32 * h, d);
      // Factored decay: one row factor (phi's scale of row r times fv or fw)
      // and one column factor cu_l = fu_l phi-scale(x_l); otherwise the cosines
      // first (bounded), then per-element exponentials of non-positive
      // arguments.
      if (!factored) {
#pragma unroll
        for (int l = 0; l < 32; ++l) d[l] = (d[l] * nr) * sc.nrm[32 * h + l];
      }
      if (r < 64) {
        // A row r: eta_r e^{g_{r-1} - g_l} <x_r, x_l> for l < r (computed, then stored)
        if (factored) {
          const float vr = nr * sc.fv[r];
#pragma unroll
          for (int l = 0; l < 32; ++l)
            d[l] = (32 * h + l < r) ? (d[l] * vr) * sc.cu[32 * h + l] : 0.f;
        } else {
          const float er = sc.eta[r], gxr = sc.gx[r];
#pragma unroll
          for (int l = 0; l < 32; ++l)
            d[l] = (32 * h + l < r) ? er * __expf(fminf(gxr - sc.g[32 * h + l], 0.f)) * d[l] : 0.f;
        }
        // A row r as bf16 for the solve's MMAs; its diagonal block (columns
        // 16 (r / 16) .. +15, in this thread's half when h == r / 32) in fp32.
        store_half_sw(a_tile, r, h, d, 1.f);
        if (h == (r >> 5)) {
          float* drow = a_diag + r * kLdD;
          if (r & 16) {
#pragma unroll
            for (int k = 0; k < 16; ++k) drow[k] = d[16 + k];
          } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) drow[k] = d[k];
          }
        }
      } else {
        // P row i: e^{g_i - g_j} <phi(q_i), x_j> for j <= i
        const int i = r - 64;
        if (factored) {
          const float wi = nr * sc.fw[i];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            d[jj] = (32 * h + jj <= i) ? (d[jj] * wi) * sc.cu[32 * h + jj] : 0.f;
        } else {
          const float gi = sc.g[i];
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            d[jj] = (32 * h + jj <= i) ? __expf(fminf(gi - sc.g[32 * h + jj], 0.f)) * d[jj] : 0.f;
        }
        store_half_sw(p_tile, i, h, d, 1.f);
      }
    }
  }
  if (__syncthreads_or(sc.fail)) goto teardown;  // A and P complete

  // ---- T' = (I + A)^{-1} Diag(eta) into the T tile (Falcon-1A: Diag(eta), written above) ----
  if (f1) solve_unit_lower_sw<true>(a_tile, a_diag, t_tile, base + L::DB, sc.eta);
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- MMA2: D[0:64) = [Xh^T; Vh^T] T^T = [W^T; U~^T] (columns of half j) ----
  if (tid == 0) {
    mma_k64(tmem, smem_addr(xh_tile), true, L::VH - L::XH, smem_addr(t_tile), false, 16,
            idesc_bf16(128, 64, true, false), false);
    mma_commit(&sc.bar_mma);
  }
  if (!wait(&sc.bar_mma, 1)) sc.fail = 1;
  tc_fence_after();
  {
    float d[32];
    tmem_ld32(tlane + 32 * h, d);
    if constexpr (kNorm) {  // column 0 of W (zero in Falcon-1A) := eta
      if (r == 0) {
#pragma unroll
        for (int l = 0; l < 32; ++l) d[l] = sc.eta[32 * h + l];
      }
    }
    store_half_sw(wu_tile, r, h, d, 1.f);  // [W^T; U~^T] over A and T (MMA2 is complete)
  }
  if (!kWide) {
    // m = 64: Xt = Diag(e^{g_C - g}) X over Xh (read by the completed MMA2),
    // and the zero tile of MMA3 over the solve's blocks in the Q tile.
    if (r < 64) store_row(xt_tile, r, 0, __expf(gC - sc.g[r]) * nr);
    reinterpret_cast<uint4*>(zero_tile)[tid] = make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4*>(zero_tile)[tid + 256] = make_uint4(0u, 0u, 0u, 0u);
  }
  // The normaliser's increment y_C over this warp's 32 rows (warps 0, 1, 4, 5):
  // the rows' scaled half rows are summed down the lanes by halving exchanges
  // (after the one over lane bit b, a lane keeps the columns whose bit b is its
  // own), which leave column 32h + lane with lane.  Rows 32..63 go through the
  // dead decay factors; rows 0..31 add them after the next barrier.
  if constexpr (kNorm) {
    if (r < 64) {
      // (the carried row x_1 = x_prev, fp32, holds zeros in xp: it is added below)
      const float s = sc.eta[r] * __expf(gC - sc.g[r]) * nr;
      float y16[16], y8[8], y4[4], y2[2];
      const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2, b0 = lane & 1;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float lo = xp.at(i) * s, hi = xp.at(i + 16) * s;
        y16[i] = (b4 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b4 ? lo : hi, 16);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        y8[i] = (b3 ? y16[i + 8] : y16[i]) +
                __shfl_xor_sync(0xffffffffu, b3 ? y16[i] : y16[i + 8], 8);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        y4[i] = (b2 ? y8[i + 4] : y8[i]) + __shfl_xor_sync(0xffffffffu, b2 ? y8[i] : y8[i + 4], 4);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        y2[i] = (b1 ? y4[i + 2] : y4[i]) + __shfl_xor_sync(0xffffffffu, b1 ? y4[i] : y4[i + 2], 2);
      ypart = (b0 ? y2[1] : y2[0]) + __shfl_xor_sync(0xffffffffu, b0 ? y2[0] : y2[1], 1);
      if (c == 0 && a.x_prev != nullptr && (warp & 1) == 0)
        ypart = fmaf(sc.eta[0] * __expf(gC - sc.g[0]), a.x_prev[bh * M + 32 * h + lane], ypart);
      if (warp & 1) sc.cu[32 * h + lane] = ypart;
    }
  }
  fence_async_smem();
  tc_fence_before();
  if (__syncthreads_or(sc.fail)) goto teardown;
  tc_fence_after();
  if constexpr (kNorm) {
    if (r < 64 && (warp & 1) == 0)
      a.norm_ws[nl.inc() + mi * 64 + 32 * h + lane] = ypart + sc.cu[32 * h + lane];
  }

  // ---- MMA3 ----
  //   m = 64:  D[0:128) = [Xt^T; 0] [W | U~] + [0; P] [W | U~]
  //   m = 128: D[0:128) = [junk; P] [W | U~] (the output rows, staged), then
  //            D[0:128) = Xt^T [W | U~] (the state rows) in the same columns
  if (tid == 0) {
    if (kWide) {
      mma_k64(tmem, smem_addr(p_tile - 8192), false, 16, smem_addr(wu_tile), false, 16,
              idesc_bf16(128, 128, false, false), false);
    } else {
      mma_k64(tmem, smem_addr(xt_tile), true, 8192, smem_addr(wu_tile), false, 16,
              idesc_bf16(128, 128, true, false), false);
      mma_k64(tmem, smem_addr(zero_tile), false, 16, smem_addr(wu_tile), false, 16,
              idesc_bf16(128, 128, false, false), true);
    }
    mma_commit(&sc.bar_mma);
  }
  if (!wait(&sc.bar_mma, 0)) sc.fail = 1;
  tc_fence_after();
  // No barrier here: each thread has seen MMA3 complete (its operands are
  // dead) before it stages; a failed wait is agreed on at the staging barrier.
  {
    unsigned char* map = reinterpret_cast<unsigned char*>(a.workspace) +
                         (size_t)(bh * nchunks + c) * L::kMapBytes;
    // The map images are staged in shared memory (the MMA3 operands are dead)
    // and leave by bulk copies.
    float d[32];
    if constexpr (!kWide) {
      unsigned char* mc_stage = kt;  // 16 KB over the K and Q tiles
      unsigned char* nc_stage = wu_tile;  // 16 KB
      // Rows 0..63 of both images come from warps 0, 1, 4, 5 and rows 64..127
      // from warps 2, 3, 6, 7: each half synchronises on its own named barrier
      // and sends its own 8 KB.
      const int grp = r >= 64 ? 1 : 0;
      const bool lead = tid == 64 * grp;  // thread 0 and thread 64
      const uint32_t half = 8192u * (uint32_t)grp;
      tmem_ld32(tlane + 32 * h, d);
      if constexpr (kNorm) {  // column 0: y_C (bf16 operands; not used) and r_t
        if (h == 0) {
          if (r >= 64) a.norm_ws[nl.rd() + mi * kC + (r - 64)] = d[0];
          d[0] = 0.f;
        }
      }
      // Mc row: rows < 64 -> -Xt^T W ; rows >= 64 -> e^{g_i} phi(q_i) - P W
      const float eq = (r >= 64) ? __expf(sc.g[r - 64]) * nr : 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) d[i] = (r < 64) ? -d[i] : eq * xp.at(i) - d[i];
      store_half_sw(mc_stage, r, h, d, 1.f);
      fence_async_smem();
      tmem_ld32(tlane + 64 + 32 * h, d);
      // (constant barrier ids in each branch: a computed id would reserve all 16)
      const bool failed = grp ? named_sync_or(2, 128, sc.fail) : named_sync_or(1, 128, sc.fail);
      // Mc leaves while Nc is staged.
      if (lead && !failed) {
        bulk_s2g_hint(map + half, mc_stage + half, kMcBytes / 2, l2_evict_last());
        bulk_commit();
      }
      store_half_sw(nc_stage, r, h, d, 1.f);  // Nc: chunk cc at position cc ^ (row & 7)
      fence_async_smem();
      if (grp)
        named_sync(2, 128);
      else
        named_sync(1, 128);
      if (lead && !failed) {
        if (grp == 0) *reinterpret_cast<float*>(map + kMcBytes + kNcBytes) = __expf(gC);
        bulk_s2g_hint(map + kMcBytes + half, nc_stage + half, kNcBytes / 2, l2_evict_last());
        bulk_commit();
        bulk_wait_read<0>();  // the staging must outlive the copies' reads
      }
    } else {
      // K-atom j of Mc (rows 0..127: -Xt^T W_j; rows 128..191: e^g phi(Q)_j - P W_j)
      // and d_v slice j of Nc (rows 0..127: Xt^T U~_j; rows 128..191: P U~_j).
      // The output rows first (lanes 64..127: P [W_j | U~_j]), staged over the
      // Xh and Vh tiles that MMA2 has read.
      unsigned char* mco_stage = xh_tile;  // 8 KB
      unsigned char* nco_stage = vh;       // 8 KB
      if (r >= 64) {  // warps 2, 3, 6, 7
        const float eq = __expf(sc.g[r - 64]) * nr;
        tmem_ld32(tlane + 32 * h, d);
#pragma unroll
        for (int i = 0; i < 32; ++i) d[i] = eq * xp.at(i) - d[i];
        store_half_sw(mco_stage, r - 64, h, d, 1.f);
        tmem_ld32(tlane + 64 + 32 * h, d);
        store_half_sw(nco_stage, r - 64, h, d, 1.f);
      }
      fence_async_smem();
      // Every thread is done with the accumulator before the state half of
      // MMA3 overwrites it.
      tc_fence_before();
      if (__syncthreads_or(sc.fail)) goto teardown;
      tc_fence_after();
      if (tid == 0) {
        mma_k64(tmem, smem_addr(xt_tile), true, L::kAtom, smem_addr(wu_tile), false, 16,
                idesc_bf16(128, 128, true, false), false);
        mma_commit(&sc.bar_mma);
      }
      if (!wait(&sc.bar_mma, 1)) sc.fail = 1;
      tc_fence_after();
      // The state rows over the operands of the completed MMA3 (Xt's first
      // atom and P; [W^T; U~^T]).
      unsigned char* mcs_stage = base;     // 16 KB
      unsigned char* ncs_stage = wu_tile;  // 16 KB
      tmem_ld32(tlane + 32 * h, d);
#pragma unroll
      for (int i = 0; i < 32; ++i) d[i] = -d[i];
      store_half_sw(mcs_stage, r, h, d, 1.f);
      tmem_ld32(tlane + 64 + 32 * h, d);
      store_half_sw(ncs_stage, r, h, d, 1.f);
      fence_async_smem();
      if (__syncthreads_or(sc.fail)) goto teardown;
      if (tid == 0) {
        unsigned char* mc = map + j * L::kMcAtom;
        unsigned char* nc = map + (2 + j) * L::kMcAtom;
        if (j == 0) *reinterpret_cast<float*>(map + 4 * L::kMcAtom) = __expf(gC);
        bulk_s2g(mc, mcs_stage, 16384);
        bulk_s2g(mc + 16384, mco_stage, 8192);
        bulk_s2g(nc, ncs_stage, 16384);
        bulk_s2g(nc + 16384, nco_stage, 8192);
        bulk_commit();
        bulk_wait_read<0>();
      }
    }
  }

teardown:
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (sc.fail && tid == 0) flag_error(err);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, L::kTmemCols);
}

// ---------------------------------------------------------------------------
// Scan kernel, one CTA per head: sixteen math warps, one issue warp and one
// refill warp.  TMEM lane rules give math warps w with (w & 3) < 2 the state
// rows (lanes 0..63) and the others the output rows (lanes 64..127); warp w
// takes columns 16 (w >> 2) .. +15 of its rows.  The state path (MMA -> state
// update -> next B operand) is the critical chain; the issue warp only waits
// and issues the MMA of each chunk, the refill warp puts the map of chunk
// c + kStages into the stage of chunk c once every math warp is done with it,
// the output rows run beside the chain, and the accumulator is
// double-buffered in TMEM.  Every hand-off is one mbarrier arrival per warp.
constexpr int kStages = kScanRing;
// The recording variant (the backward's recomputed forward: no o, the state
// entering every chunk written out) keeps four stages and no o staging.
constexpr int kRecStages = 4;
constexpr int kScanMathWarps = 16;
constexpr int kScanThreads = 32 * (kScanMathWarps + 2);

template <int kSt, bool kOut>
struct ScanSmemT {
  unsigned char mc[kSt][kMcBytes];  // A tiles of the state MMA (K-major)
  unsigned char nc[kSt][kNcBytes];  // Nc rows (bf16, 16-byte chunks swizzled)
  unsigned char sop[8192];          // S as MN-major B operand (rows = m, 64 bf16 along d_v)
  unsigned char ostage[kOut ? 2 : 1][kOut ? 8192 : 16];  // o tiles (64 x 64 bf16) for TMA
  float gc[kSt][4];
  uint64_t full[kSt];   // map of the stage has arrived
  uint64_t empty[kSt];  // every math warp is done with the stage
  uint64_t mma_done[2];     // MMA into accumulator buffer b has completed
  uint64_t o_done[2];       // output warps have read accumulator buffer b
  uint64_t s_ready;         // the next state operand is in sop
  uint32_t tmem_base;
  int fail;
};
using ScanSmem = ScanSmemT<kStages, true>;
using RecScanSmem = ScanSmemT<kRecStages, false>;

template <typename Smem>
__device__ __forceinline__ void issue_map_load(Smem& s, int st, const unsigned char* m) {
  mbar_expect_tx(&s.full[st], kMcBytes + kNcBytes + 16);
  const uint64_t pol = l2_evict_first();
  bulk_g2s_hint(s.mc[st], m, kMcBytes, &s.full[st], pol);
  bulk_g2s_hint(s.nc[st], m + kMcBytes, kNcBytes, &s.full[st], pol);
  bulk_g2s(s.gc[st], m + kMcBytes + kNcBytes, 16, &s.full[st]);
}

// Sixteen bf16 values (two 16-byte chunks) added to d.
__device__ __forceinline__ void add_bf16x16(float* d, uint4 p0, uint4 p1) {
  const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&p0);
  const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&p1);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f0 = __bfloat1622float2(h0[e]);
    const float2 f1 = __bfloat1622float2(h1[e]);
    d[2 * e] += f0.x;
    d[2 * e + 1] += f0.y;
    d[8 + 2 * e] += f1.x;
    d[8 + 2 * e + 1] += f1.y;
  }
}

// kRecord: write the state entering every chunk to a.S_starts and no o (the
// output warps stay idle; four map stages).
template <bool kRecord>
__global__ void __launch_bounds__(kScanThreads, 1)
    tc_chunk_scan_kernel(ChunkArgs a, int nchunks, int c_begin, int n, const float* S_in, int* err,
                         const __grid_constant__ CUtensorMap tm_o) {
  using Smem = std::conditional_t<kRecord, RecScanSmem, ScanSmem>;
  constexpr int kSt = kRecord ? kRecStages : kStages;
  extern __shared__ unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(align1024(smem_raw));
  volatile int* fail = &s.fail;
  const int64_t bh = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool issuer = warp == kScanMathWarps;
  const bool refiller = warp == kScanMathWarps + 1;
  const int row = 32 * (warp & 3) + lane;  // TMEM lane = row of [S'; O]
  const int qc = (warp >> 2) & 3;          // column quarter: 16 qc .. 16 qc + 15
  const bool srow = warp < kScanMathWarps && row < 64;
  // The two 16-byte chunks of this thread's columns, at their swizzled places.
  const uint32_t ch0 = (uint32_t)(((2 * qc) ^ (row & 7)) << 4);
  const uint32_t ch1 = (uint32_t)(((2 * qc + 1) ^ (row & 7)) << 4);
  const unsigned char* ws = reinterpret_cast<const unsigned char*>(a.workspace) +
                            ((size_t)bh * nchunks + c_begin) * kMapBytes;  // this range's maps
  // A following map launch may start now; it waits for this grid to complete
  // before it touches memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 0) tmem_alloc(&s.tmem_base, 128);
  if (tid == 0) {
    for (int st = 0; st < kSt; ++st) {
      mbar_init(&s.full[st], 1);
      mbar_init(&s.empty[st], kRecord ? kScanMathWarps / 2 : kScanMathWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.mma_done[b], 1);
      mbar_init(&s.o_done[b], kScanMathWarps / 2);
    }
    mbar_init(&s.s_ready, kScanMathWarps / 2);
    fence_mbar_init();
    s.fail = 0;
  }
  // State: each state thread keeps 16 columns of its row in fp32 registers.
  float S[16];
  if (srow) {
#pragma unroll
    for (int j = 0; j < 16; ++j) S[j] = S_in ? S_in[(bh * 64 + row) * 64 + 16 * qc + j] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The maps are written by the preceding launch: wait for it to complete.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tmem = s.tmem_base;

  if (issuer) {
    if (lane == 0) {
      for (int st = 0; st < kSt && st < n; ++st)
        issue_map_load(s, st, ws + (size_t)st * kMapBytes);
      const uint64_t bdesc = sw128_desc(smem_addr(s.sop), 8192, 1024);
      const uint32_t idesc = idesc_bf16(128, 64, false, true);
      for (int c = 0; c < n; ++c) {
        const int st = c % kSt, b = c & 1;
        // The state operand is the last to be ready: wait for it last.  (The
        // state rows of accumulator b were read before the operand of chunk
        // c - 1 was signalled; without o nothing else reads it.)
        bool ok = kRecord || c < 2 || mbar_wait(&s.o_done[b], (uint32_t)((c - 2) >> 1) & 1u);
        ok = ok && mbar_wait(&s.full[st], (uint32_t)(c / kSt) & 1u);
        ok = ok && mbar_wait(&s.s_ready, (uint32_t)c & 1u);
        if (!ok) {
          *fail = 1;
          break;
        }
        tc_fence_after();
        mma_k64_desc(tmem + 64 * b, sw128_desc(smem_addr(s.mc[st]), 16, 1024), kStepK, bdesc,
                     kStepMN, idesc, false);
        mma_commit(&s.mma_done[b]);
      }
    }
    __syncwarp();
  } else if (refiller) {
    // The stage of chunk c gets chunk c + kSt once every math warp is done
    // with it (the MMA of chunk c has then completed too).
    if (lane == 0) {
      for (int c = 0; c + kSt < n; ++c) {
        if (*fail) break;
        const int st = c % kSt;
        if (!mbar_wait(&s.empty[st], (uint32_t)(c / kSt) & 1u)) {
          *fail = 1;
          break;
        }
        issue_map_load(s, st, ws + (size_t)(c + kSt) * kMapBytes);
      }
    }
    __syncwarp();
  } else if (srow) {
    // ---- state warps: the critical chain ----
    const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 16 * qc;
    *reinterpret_cast<uint4*>(s.sop + row * 128 + ch0) = pack8(S, 1.f);
    *reinterpret_cast<uint4*>(s.sop + row * 128 + ch1) = pack8(S + 8, 1.f);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.s_ready);
    for (int c = 0; c < n; ++c) {
      // Exits are warp-uniform, so every __syncwarp sees all lanes.
      if (__any_sync(0xffffffffu, *fail)) break;
      if (kRecord) {  // the state entering chunk c (for the backward pass)
        float4* dst = reinterpret_cast<float4*>(
            a.S_starts + (((size_t)bh * nchunks + c_begin + c) * 64 + row) * 64 + 16 * qc);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          dst[q4] = make_float4(S[4 * q4], S[4 * q4 + 1], S[4 * q4 + 2], S[4 * q4 + 3]);
      }
      const int st = c % kSt, b = c & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&s.full[st], (uint32_t)(c / kSt) & 1u))) {
        *fail = 1;
        break;
      }
      // Nc (this thread's 16 columns) and e^{g_C} before the MMA completes.
      const unsigned char* nrow = s.nc[st] + row * 128;
      const uint4 n0 = *reinterpret_cast<const uint4*>(nrow + ch0);
      const uint4 n1 = *reinterpret_cast<const uint4*>(nrow + ch1);
      const float gC = s.gc[st][0];
      if (!__all_sync(0xffffffffu, mbar_wait(&s.mma_done[b], (uint32_t)(c >> 1) & 1u))) {
        *fail = 1;
        break;
      }
      tc_fence_after();
      float d[16];
      tmem_ld16(tlane + 64 * b, d);
      tc_fence_before();
      add_bf16x16(d, n0, n1);
#pragma unroll
      for (int j = 0; j < 16; ++j) S[j] = gC * S[j] + d[j];
      *reinterpret_cast<uint4*>(s.sop + row * 128 + ch0) = pack8(S, 1.f);
      *reinterpret_cast<uint4*>(s.sop + row * 128 + ch1) = pack8(S + 8, 1.f);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s.s_ready);
        mbar_arrive(&s.empty[st]);  // Nc read; the MMA has read Mc
      }
    }
  } else if constexpr (!kRecord) {
    // ---- output warps: o rows, off the chain.  The o tile of a chunk leaves
    // by one TMA store issued by the first lane of warp 2; rows past T are
    // dropped by the tensor map.  Exits are agreed on by all output warps at
    // a named barrier, so none is left waiting there.
    const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 16 * qc;
    const bool o_issuer = warp == 2 && lane == 0;
    constexpr int kOutThreads = 32 * kScanMathWarps / 2;
    for (int c = 0; c < n; ++c) {
      const int st = c % kSt, b = c & 1;
      bool ok = !*fail && mbar_wait(&s.full[st], (uint32_t)(c / kSt) & 1u);
      uint4 n0 = make_uint4(0u, 0u, 0u, 0u), n1 = n0;
      if (ok) {
        const unsigned char* nrow = s.nc[st] + row * 128;
        n0 = *reinterpret_cast<const uint4*>(nrow + ch0);
        n1 = *reinterpret_cast<const uint4*>(nrow + ch1);
      }
      ok = ok && mbar_wait(&s.mma_done[b], (uint32_t)(c >> 1) & 1u);
      // Staging buffer b was last read by the TMA store of chunk c - 2.
      if (o_issuer) bulk_wait_read<1>();
      if (named_sync_or(1, kOutThreads, !ok)) {
        *fail = 1;
        break;
      }
      tc_fence_after();
      float d[16];
      tmem_ld16(tlane + 64 * b, d);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s.o_done[b]);  // accumulator b is read
        mbar_arrive(&s.empty[st]);  // Nc read; the MMA has read Mc
      }
      add_bf16x16(d, n0, n1);
      unsigned char* orow = s.ostage[b] + (row - 64) * 128;
      *reinterpret_cast<uint4*>(orow + ch0) = pack8(d, 1.f);
      *reinterpret_cast<uint4*>(orow + ch1) = pack8(d + 8, 1.f);
      fence_async_smem();
      named_sync(1, kOutThreads);
      if (o_issuer) {
        tma_store_3d(&tm_o, s.ostage[b], 0, (c_begin + c) * kC, (int)bh);
        bulk_commit();
      }
    }
    if (o_issuer) bulk_wait<0>();  // the o stores have landed
  }
  if (!*fail && srow)
#pragma unroll
    for (int j = 0; j < 16; ++j) a.S_out[(bh * 64 + row) * 64 + 16 * qc + j] = S[j];
  __syncthreads();
  if (*fail && tid == 0) flag_error(err);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
// Scan kernel for m = d_v = 128: one CTA per (head, d_v slice j of 64
// columns); the slices are independent (the map acts on each column of S).
// Per chunk two MMAs read the same state operand S_j (128 x 64, bf16): rows
// 0..127 of Mc (the state rows, K = 128 over two K-atoms) and rows 128..255
// (the 64 output rows, then 64 rows past the map that land in unused
// accumulator lanes).  Warps 0..15 own the state rows (lane quarter w & 3,
// columns 16 (w >> 2) .. +15), warps 16, 17, 20, 21 the output rows (lane
// quarters 0 and 1, column halves).  Warp 18 issues the MMAs: per chunk the
// state MMA (committed on its own barrier, so the state chain does not wait
// for the output rows), then the output MMA, which runs on the tensor pipe
// while the state warps update S.  Warp 19 refills the map ring, so the
// issuing thread waits only for what the next MMA reads.
// The Mc atoms go through a three-stage shared-memory ring; Nc rows are read
// from global memory (brought into L2 ahead by the refill warp) one chunk ahead
// into registers, which keeps three map stages within shared memory.
constexpr int kStages128 = 3;
constexpr int kScan128Threads = 32 * 22;
constexpr uint32_t kStage128Bytes = 49 * 1024;  // Mc atoms (2 x 24 KB), e^{g_C}

struct Scan128Smem {
  unsigned char stage[kStages128][kStage128Bytes];
  // S_j as MN-major B operand (128 rows = m, 64 bf16 along d_v), double-buffered:
  // chunk c reads sop[c & 1] while the state warps write S_{c+1} to the other
  // buffer (the output MMAs of chunk c may still be reading it).
  unsigned char sop[2][16384];
  unsigned char ostage[2][8192];   // o tiles (64 tokens x 64 bf16, 128B-swizzled) for TMA
  uint64_t full[kStages128];       // map of the stage has arrived
  uint64_t empty[kStages128];      // every math warp is done with the stage
  uint64_t mma_done[2];            // state MMAs into accumulator buffer b have completed
  uint64_t omma_done[2];           // output MMAs into accumulator buffer b have completed
  uint64_t o_done[2];              // output warps have read accumulator buffer b
  uint64_t s_ready;                // the next state operand is in sop
  uint32_t tmem_base;
  int fail;
};

__device__ __forceinline__ void issue_map_load128(Scan128Smem& s, int st, const unsigned char* m,
                                                  int j) {
  constexpr uint32_t kA = MapLayout<128>::kMcAtom;
  unsigned char* dst = s.stage[st];
  mbar_expect_tx(&s.full[st], 2 * kA + 16);
  bulk_g2s(dst, m, kA, &s.full[st]);
  bulk_g2s(dst + kA, m + kA, kA, &s.full[st]);
  bulk_g2s(dst + 2 * kA, m + 4 * kA, 16, &s.full[st]);
  bulk_prefetch_l2(m + (2 + j) * kA, kA);  // this CTA's Nc slice
}

// 16 bytes of the (read-only) workspace.
__device__ __forceinline__ uint4 ld_map16(const unsigned char* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__global__ void __launch_bounds__(kScan128Threads)
    tc_chunk_scan128_kernel(ChunkArgs a, int nchunks, int c_begin, int n, const float* S_in,
                            int* err,
                            const __grid_constant__ CUtensorMap tm_o) {
  constexpr uint32_t kA = MapLayout<128>::kMcAtom;
  constexpr uint32_t kMap = MapLayout<128>::kMapBytes;
  constexpr int kOutWarps = 4;
  extern __shared__ unsigned char smem_raw[];
  Scan128Smem& s = *reinterpret_cast<Scan128Smem*>(align1024(smem_raw));
  volatile int* fail = &s.fail;
  const int64_t bh = blockIdx.x >> 1;
  const int j = blockIdx.x & 1;  // d_v slice
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool issuer = warp == 18;
  const bool refiller = warp == 19;
  const bool swarp = warp < 16;
  const bool owarp = warp == 16 || warp == 17 || warp == 20 || warp == 21;
  const int row = 32 * (warp & 3) + lane;  // TMEM lane
  const unsigned char* ws = reinterpret_cast<const unsigned char*>(a.workspace) +
                            ((size_t)bh * nchunks + c_begin) * kMap;  // this range's maps
  // A following map launch may start now; it waits for this grid to complete
  // before it touches memory.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 0) tmem_alloc(&s.tmem_base, 256);
  if (tid == 0) {
    for (int st = 0; st < kStages128; ++st) {
      mbar_init(&s.full[st], 1);
      mbar_init(&s.empty[st], 16 + kOutWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.mma_done[b], 1);
      mbar_init(&s.omma_done[b], 1);
      mbar_init(&s.o_done[b], kOutWarps);
    }
    mbar_init(&s.s_ready, 16);
    fence_mbar_init();
    s.fail = 0;
  }
  // State: each state thread keeps 16 columns of its row in fp32 registers.
  const int qc = (warp >> 2) & 3;  // state warps: column quarter
  float S[16];
  if (swarp) {
    const float* src = S_in ? S_in + (bh * 128 + row) * 128 + 64 * j + 16 * qc : nullptr;
#pragma unroll
    for (int i = 0; i < 16; ++i) S[i] = src ? src[i] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tmem = s.tmem_base;

  if (issuer) {
    if (lane == 0) {
      for (int st = 0; st < kStages128 && st < n; ++st)
        issue_map_load128(s, st, ws + (size_t)st * kMap, j);
      const uint32_t idesc = idesc_bf16(128, 64, false, true);
      for (int c = 0; c < n; ++c) {
        const int st = c % kStages128, b = c & 1;
        // Accumulator buffer b free (output rows of chunk c - 2 read), the map
        // in its stage; the state operand is the last to be ready: wait for it last.
        bool ok = c < 2 || mbar_wait(&s.o_done[b], (uint32_t)((c - 2) >> 1) & 1u);
        ok = ok && mbar_wait(&s.full[st], (uint32_t)(c / kStages128) & 1u);
        ok = ok && mbar_wait(&s.s_ready, (uint32_t)c & 1u);
        if (!ok) {
          *fail = 1;
          break;
        }
        tc_fence_after();
        // State rows, K = 128 as two 64-wide atoms.
        const uint64_t ad = sw128_desc(smem_addr(s.stage[st]), 16, 1024);
        const uint64_t bdesc0 = sw128_desc(smem_addr(s.sop[c & 1]), 8192, 1024);
        const uint64_t bdesc1 = bdesc0 + (8192 >> 4);  // state rows 64..127
        mma_k64_desc(tmem + 128 * b, ad, kStepK, bdesc0, kStepMN, idesc, false);
        mma_k64_desc(tmem + 128 * b, ad + (kA >> 4), kStepK, bdesc1, kStepMN, idesc, true);
        mma_commit(&s.mma_done[b]);
        // Output rows (Mc rows 128..255), same operand.
        mma_k64_desc(tmem + 128 * b + 64, ad + (16384 >> 4), kStepK, bdesc0, kStepMN, idesc,
                     false);
        mma_k64_desc(tmem + 128 * b + 64, ad + ((kA + 16384) >> 4), kStepK, bdesc1, kStepMN,
                     idesc, true);
        mma_commit(&s.omma_done[b]);
      }
    }
    __syncwarp();
  } else if (refiller) {
    // The stage of chunk c gets chunk c + kStages128 once every math warp is
    // done with it (both MMAs of chunk c have then completed too).
    if (lane == 0) {
      for (int c = 0; c + kStages128 < n; ++c) {
        if (*fail) break;
        const int st = c % kStages128;
        if (!mbar_wait(&s.empty[st], (uint32_t)(c / kStages128) & 1u)) {
          *fail = 1;
          break;
        }
        issue_map_load128(s, st, ws + (size_t)(c + kStages128) * kMap, j);
      }
    }
    __syncwarp();
  } else if (swarp) {
    const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 16 * qc;
    const uint32_t ch0 = (uint32_t)(((2 * qc) ^ (row & 7)) << 4);
    const uint32_t ch1 = (uint32_t)(((2 * qc + 1) ^ (row & 7)) << 4);
    *reinterpret_cast<uint4*>(s.sop[0] + row * 128 + ch0) = pack8(S, 1.f);
    *reinterpret_cast<uint4*>(s.sop[0] + row * 128 + ch1) = pack8(S + 8, 1.f);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.s_ready);
    // Nc rows of this thread (state rows 0..127 of slice j), one chunk ahead
    // of their use.  The loop runs two chunks per pass so that the rows of the
    // next chunk land in the other register pair, with no copy that would
    // wait for the load on the chain.
    const unsigned char* ncg = ws + (2 + j) * kA + row * 128;
    uint4 na0 = ld_map16(ncg + ch0), na1 = ld_map16(ncg + ch1);
    uint4 nb0 = make_uint4(0u, 0u, 0u, 0u), nb1 = nb0;
    // One chunk: uses (cur0, cur1), loads chunk c + 1 into (nxt0, nxt1).
    auto chunk_step = [&](int c, const uint4& cur0, const uint4& cur1, uint4& nxt0,
                          uint4& nxt1) -> bool {
      if (__any_sync(0xffffffffu, *fail)) return false;
      const int st = c % kStages128, b = c & 1;
      // mma_done of chunk c also covers the MMAs of chunk c - 1 (issued
      // earlier by the same thread), the last readers of sop[(c + 1) & 1].
      unsigned char* sop_next = s.sop[(c + 1) & 1];
      if (!__all_sync(0xffffffffu, mbar_wait(&s.full[st], (uint32_t)(c / kStages128) & 1u))) {
        *fail = 1;
        return false;
      }
      const float gC = *reinterpret_cast<const float*>(s.stage[st] + 2 * kA);
      if (c + 1 < n) {
        const unsigned char* nrow = ncg + (size_t)(c + 1) * kMap;
        nxt0 = ld_map16(nrow + ch0);
        nxt1 = ld_map16(nrow + ch1);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&s.mma_done[b], (uint32_t)(c >> 1) & 1u))) {
        *fail = 1;
        return false;
      }
      tc_fence_after();
      float d[16];
      tmem_ld16(tlane + 128 * b, d);
      tc_fence_before();
      add_bf16x16(d, cur0, cur1);
#pragma unroll
      for (int i = 0; i < 16; ++i) S[i] = gC * S[i] + d[i];
      *reinterpret_cast<uint4*>(sop_next + row * 128 + ch0) = pack8(S, 1.f);
      *reinterpret_cast<uint4*>(sop_next + row * 128 + ch1) = pack8(S + 8, 1.f);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s.s_ready);
        mbar_arrive(&s.empty[st]);
      }
      return true;
    };
    for (int c = 0; c < n; c += 2) {
      if (!chunk_step(c, na0, na1, nb0, nb1)) break;
      if (c + 1 < n && !chunk_step(c + 1, nb0, nb1, na0, na1)) break;
    }
    if (!*fail) {
      float* dst = a.S_out + (bh * 128 + row) * 128 + 64 * j + 16 * qc;
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i] = S[i];
    }
  } else if (owarp) {
    // Output rows 0..63 (lanes 0..63 of the second accumulator), 32 columns
    // per thread; the o tile leaves by one TMA store per chunk (warp 16, lane
    // 0); exits are agreed on by the output warps at a named barrier.
    const int oh = (warp - 16) >> 2;  // column half: 32 oh .. 32 oh + 31
    const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 + 32 * oh;
    const bool o_issuer = warp == 16 && lane == 0;
    // Nc rows 128 + row (the output rows of slice j), one chunk ahead.
    const unsigned char* ncg = ws + (2 + j) * kA + (128 + row) * 128;
    // Two chunks per pass, so the rows of the next chunk land in the other
    // register set with no copy that would wait for the load.
    uint4 na[4], nb[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      na[q] = ld_map16(ncg + (((4 * oh + q) ^ (row & 7)) << 4));
      nb[q] = make_uint4(0u, 0u, 0u, 0u);
    }
    // One chunk: uses cur, loads the rows of chunk c + 1 into nxt.
    auto out_step = [&](int c, const uint4 (&cur)[4], uint4 (&nxt)[4]) -> bool {
      const int st = c % kStages128, b = c & 1;
      if (c + 1 < n) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          nxt[q] = ld_map16(ncg + (size_t)(c + 1) * kMap + (((4 * oh + q) ^ (row & 7)) << 4));
      }
      bool ok = !*fail && mbar_wait(&s.full[st], (uint32_t)(c / kStages128) & 1u);
      ok = ok && mbar_wait(&s.omma_done[b], (uint32_t)(c >> 1) & 1u);
      if (o_issuer) bulk_wait_read<1>();
      if (named_sync_or(1, 32 * kOutWarps, !ok)) {
        *fail = 1;
        return false;
      }
      tc_fence_after();
      float d[32];
      tmem_ld32(tlane + 128 * b, d);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s.o_done[b]);  // accumulator b is read
        mbar_arrive(&s.empty[st]);  // the MMAs of chunk c have read its stage
      }
      // + Nc rows 128.. (output rows), this thread's four 16-byte chunks
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&cur[q]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(hv[e]);
          d[8 * q + 2 * e] += f.x;
          d[8 * q + 2 * e + 1] += f.y;
        }
      }
      unsigned char* orow = s.ostage[b] + row * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(orow + (((4 * oh + q) ^ (row & 7)) << 4)) = pack8(d + 8 * q, 1.f);
      fence_async_smem();
      named_sync(1, 32 * kOutWarps);
      if (o_issuer) {
        tma_store_3d(&tm_o, s.ostage[b], 64 * j, (c_begin + c) * kC, (int)bh);
        bulk_commit();
      }
      return true;
    };
    for (int c = 0; c < n; c += 2) {
      if (!out_step(c, na, nb)) break;
      if (c + 1 < n && !out_step(c + 1, nb, na)) break;
    }
    if (o_issuer) bulk_wait<0>();
  }
  __syncthreads();
  if (*fail && tid == 0) flag_error(err);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace

bool tc_path_applies(int dtype, int m, int dv, int C, int64_t BH, int64_t T) {
  // TMA box coordinates are 32-bit: rows and heads stay below 2^31.
  return dtype == FALCON_BF16 && (m == 64 || m == 128) && dv == m && C == 64 &&
         T < (int64_t(1) << 31) - kC && BH < (int64_t(1) << 30);
}

size_t tc_workspace_bytes(int m, int64_t BH, int64_t T) {
  const int64_t nch = (T + kC - 1) / kC;
  return (size_t)(BH * nch) * (m == 128 ? MapLayout<128>::kMapBytes : MapLayout<64>::kMapBytes);
}

namespace {

// CTAs of tc_chunk_map_kernel<M> resident on the current device at once (SMs x
// CTAs per SM), cached per device; 0 if the runtime cannot tell (no prefetch).
template <int M>
uint32_t map_residency() {
  static std::atomic<uint32_t> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  uint32_t v = cache[dev].load(std::memory_order_relaxed);
  if (v != 0) return v;
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_chunk_map_kernel<M>, kMapThreads,
                                                    map_smem_bytes<M>() + 1024) != cudaSuccess)
    return 0;
  v = (uint32_t)(sms > 0 ? sms : 0) * (uint32_t)(per_sm > 0 ? per_sm : 0);
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// pdl: programmatic dependent launch behind the preceding kernel on the stream
// (the map kernel waits for it with griddepcontrol.wait before reading inputs).
template <int M>
cudaError_t launch_map(const ChunkArgs& a, int nchunks, int c_begin, int n, int* err,
                       const CUtensorMap& tm_k, const CUtensorMap& tm_q, const CUtensorMap& tm_v,
                       bool pdl, cudaStream_t stream) {
  const size_t smem = map_smem_bytes<M>() + 1024;
  // The variant that also writes the normalised read's per-chunk terms (m = 64).
  auto kernel = tc_chunk_map_kernel<M, false>;
  if constexpr (M == 64) {
    if (a.norm_ws && a.rule == kFalcon1A) kernel = tc_chunk_map_kernel<64, true>;
  }
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n * MapLayout<M>::kHalves, (unsigned)a.BH);
  cfg.blockDim = dim3(kMapThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, a, nchunks, c_begin, err, map_residency<M>(), tm_k,
                            tm_q, tm_v);
}

// pdl: programmatic dependent launch after the preceding map launch on the
// same stream (griddepcontrol.wait in the scan orders it after every map write).
template <typename Kernel>
cudaError_t launch_scan(Kernel kernel, unsigned grid, unsigned threads, size_t smem, bool pdl,
                        const ChunkArgs& a, int nchunks, int c_begin, int n, const float* S_in,
                        int* err, const CUtensorMap& tm_o, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, a, nchunks, c_begin, n, S_in, err, tm_o);
}

// Pieces of the chunk range: with few heads and many chunks the scan runs on
// few SMs for a long time, so the call is cut into chunk ranges whose scans run
// on a second stream while the maps of the next range run on the caller's
// stream (event-ordered; no kernel waits on another).  The second stream has
// the highest priority, so the CTAs of a pending scan (the sequential part,
// which bounds the call) are placed ahead of the next range's map CTAs.  With
// many heads the scan already fills most SMs and a single range is kept
// (measured on the lm shape: 1 range 118 us, 2 ranges 136 us).  Long shape,
// 1024 chunks of 16 heads, side stream at the default priority: 1, 4, 8, 16,
// 32 ranges took 2.65, 2.18, 1.94, 1.90, 2.06 ms; with the current map kernel
// and the side stream at the highest priority, 8, 16, 32 ranges took 1.75,
// 1.84, 2.09 ms.
int piece_count(int64_t BH, int nchunks, bool wide) {
  const int64_t scan_ctas = BH * (wide ? 2 : 1);
  if (scan_ctas > 64 || nchunks < 64) return 1;
  return nchunks >= 256 ? 8 : 4;
}

constexpr int kMaxPieces = 16;
constexpr int kMaxDevices = 64;

// Per-device second stream and events (created once, on first use).
struct PieceStreams {
  cudaStream_t side = nullptr;
  cudaEvent_t map_done[kMaxPieces] = {};
  cudaEvent_t scans_done = nullptr;
  bool ready = false;
};
std::mutex g_piece_mu;
PieceStreams g_piece[kMaxDevices];

cudaError_t piece_streams(PieceStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  PieceStreams& ps = g_piece[dev];
  if (!ps.ready) {
    int least = 0, greatest = 0;
    if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithPriority(&ps.side, cudaStreamNonBlocking, greatest)) !=
        cudaSuccess)
      return e;
    for (int i = 0; i < kMaxPieces; ++i)
      if ((e = cudaEventCreateWithFlags(&ps.map_done[i], cudaEventDisableTiming)) != cudaSuccess)
        return e;
    if ((e = cudaEventCreateWithFlags(&ps.scans_done, cudaEventDisableTiming)) != cudaSuccess)
      return e;
    ps.ready = true;
  }
  *out = &ps;
  return cudaSuccess;
}

template <int M>
cudaError_t launch_scan_range(const ChunkArgs& a, int nchunks, int c_begin, int n,
                              const float* S_in, bool pdl, int* err, const CUtensorMap& tm_o,
                              cudaStream_t stream) {
  if (M == 128)
    return launch_scan(tc_chunk_scan128_kernel, (unsigned)(2 * a.BH), kScan128Threads,
                       sizeof(Scan128Smem) + 1024, pdl, a, nchunks, c_begin, n, S_in, err, tm_o,
                       stream);
  if (a.S_starts)
    return launch_scan(tc_chunk_scan_kernel<true>, (unsigned)a.BH, kScanThreads,
                       sizeof(RecScanSmem) + 1024, pdl, a, nchunks, c_begin, n, S_in, err, tm_o,
                       stream);
  return launch_scan(tc_chunk_scan_kernel<false>, (unsigned)a.BH, kScanThreads,
                     sizeof(ScanSmem) + 1024, pdl, a, nchunks, c_begin, n, S_in, err, tm_o,
                     stream);
}

template <int M>
cudaError_t launch_tc(const ChunkArgs& a, int* err, cudaStream_t stream) {
  const int nchunks = (int)((a.T + kC - 1) / kC);
  CUtensorMap tm_k, tm_q, tm_v, tm_o;
  if (!encode_rows_bf16(&tm_k, a.k, M, (uint64_t)a.T, (uint64_t)a.BH, 64, kC) ||
      !encode_rows_bf16(&tm_q, a.q, M, (uint64_t)a.T, (uint64_t)a.BH, 64, kC) ||
      !encode_rows_bf16(&tm_v, a.v, M, (uint64_t)a.T, (uint64_t)a.BH, 64, kC) ||
      !encode_rows_bf16(&tm_o, a.o, M, (uint64_t)a.T, (uint64_t)a.BH, 64, kC))
    return cudaErrorInvalidValue;
  const int pieces = piece_count(a.BH, nchunks, M == 128);
  if (pieces == 1) {
    cudaError_t e = launch_map<M>(a, nchunks, 0, nchunks, err, tm_k, tm_q, tm_v, true, stream);
    if (e != cudaSuccess) return e;
    return launch_scan_range<M>(a, nchunks, 0, nchunks, a.S0, true, err, tm_o, stream);
  }
  // The scans of consecutive ranges run in order on the side stream, each after
  // its range's maps; the running state goes through S_out (S_out may alias
  // S0: a scan reads its initial state before writing the same elements).
  std::lock_guard<std::mutex> lock(g_piece_mu);
  PieceStreams* ps = nullptr;
  cudaError_t e = piece_streams(&ps);
  if (e != cudaSuccess) return e;
  for (int p = 0; p < pieces; ++p) {
    const int c0 = (int)((int64_t)nchunks * p / pieces);
    const int c1 = (int)((int64_t)nchunks * (p + 1) / pieces);
    if ((e = launch_map<M>(a, nchunks, c0, c1 - c0, err, tm_k, tm_q, tm_v, false, stream)) !=
        cudaSuccess)
      return e;
    if ((e = cudaEventRecord(ps->map_done[p], stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ps->side, ps->map_done[p], 0)) != cudaSuccess) return e;
    e = launch_scan_range<M>(a, nchunks, c0, c1 - c0, p == 0 ? a.S0 : a.S_out, false, err, tm_o,
                             ps->side);
    if (e != cudaSuccess) return e;
  }
  if ((e = cudaEventRecord(ps->scans_done, ps->side)) != cudaSuccess) return e;
  return cudaStreamWaitEvent(stream, ps->scans_done, 0);
}

}  // namespace

cudaError_t launch_tc_scan64(const ChunkArgs& a, int* err, cudaStream_t stream) {
  const int nchunks = (int)((a.T + kC - 1) / kC);
  CUtensorMap tm_o;
  if (!encode_rows_bf16(&tm_o, a.o, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kC))
    return cudaErrorInvalidValue;
  return launch_scan_range<64>(a, nchunks, 0, nchunks, a.S0, true, err, tm_o, stream);
}

cudaError_t launch_tc_chunked(const ChunkArgs& a, int* err, cudaStream_t stream) {
  return a.m == 128 ? launch_tc<128>(a, err, stream) : launch_tc<64>(a, err, stream);
}

cudaError_t launch_tc_map64(const ChunkArgs& a, int* err, cudaStream_t stream) {
  const int nchunks = (int)((a.T + kC - 1) / kC);
  CUtensorMap tm_k, tm_q, tm_v;
  if (!encode_rows_bf16(&tm_k, a.k, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kC) ||
      !encode_rows_bf16(&tm_q, a.q, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kC) ||
      !encode_rows_bf16(&tm_v, a.v, 64, (uint64_t)a.T, (uint64_t)a.BH, 64, kC))
    return cudaErrorInvalidValue;
  return launch_map<64>(a, nchunks, 0, nchunks, err, tm_k, tm_q, tm_v, true, stream);
}


}  // namespace falcon
