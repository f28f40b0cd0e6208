// Chunked path of the gated delta rule on sm_103a tensor cores (tcgen05 +
// TMEM + TMA), chunk size C = 64.
//
// Within a chunk of C tokens that starts from state S0 (d_v x d_k, stored
// [value][key]), with G_r the running sum of g inside the chunk (inclusive),
// gamma_r = exp(G_r) and u_r = beta_r (v_r - exp(g_r) S_{r-1} k_r) the
// correction token r writes, the recurrence unrolls to
//     S_r = gamma_r S0 + sum_{i<=r} exp(G_r - G_i) u_i k_i^T,
// and the corrections solve a unit lower-triangular system
//     (I + A) U = R,   A[r,i] = beta_r exp(G_r - G_i) (k_r . k_i)  (i < r)
//                      R = diag(beta) V - diag(beta gamma) K S0^T.
// With T = (I + A)^-1 (the UT transform of the chunk) and the causal decay
// mask P[r,i] = exp(G_r - G_i) (q_r . k_i) (i <= r):
//     U = T R,   O = (diag(gamma) Q S0^T + P U) / sqrt(d),
//     S_C = gamma_{C-1} S0 + (diag(exp(G_{C-1} - G)) U)^T K.
// "Gated Delta Net on AMD: why ROCm stumbles on hybrid-attention LLMs",
// section "Why this bites AMD users specifically": the chunked form turns the
// sequential recurrence into blocks that run in parallel; "marcsun13/
// ggml-gated-delta-net" model card, section "Ops": one dispatch per run of
// steps, state [value][key], 1/sqrt(head_dim) output scale, log-domain gate.
//
// GB300 mapping.  The chunk transform Z = [T; P T] (128 x 64) depends on
// K, Q and the gates only; the state walk needs Z and the state.  Three
// kernels share the steps below:
//   - chunked_d128_kernel (head_dim 64 and 128): one CTA per (sequence,
//     head) holds the whole state in TMEM, value rows on lanes, and runs
//     two warp-specialised streams: 8 warps build Z one chunk ahead, 8 warps
//     walk the state.
//   - chunk_z_kernel + chunked_kernel (head_dim 256, and head_dim 128 with
//     few (sequence, head) pairs): persistent CTAs write every chunk's Z to
//     a workspace; the state walk (a dependent launch that starts while the
//     transform finishes) then runs one CTA per block of 64 value rows (32
//     where that still fits the pairs into one wave of CTAs, or for the
//     pairs past the last full wave of 64-row blocks), keys on lanes, the
//     fp32 state in registers.
// Per chunk:
//   1. TMA (128-byte swizzle) brings K, Q (stacked as one 128-row tile) and
//      V; plain loads bring g, beta.
//   2. MMA  [K;Q] K^T -> TMEM (M=128, N=64): K K^T and Q K^T in one tile.
//   3. A and P from it; T = (I + A)^-1 by 32x32 or 16x16 blocks (diagonal
//      blocks on CUDA cores, block products on warp-level MMAs); MMA  P T; the
//      stacked Z = [T; P T] is written as bf16 hi + lo (two bf16 terms).
//   4. MMA  [K;Q] S0^T -> TMEM: both K S0^T (for R) and Q S0^T (for O).
//   5. R = beta V - beta gamma K S0^T, written as bf16 hi + lo.
//   6. MMA  Z R -> TMEM: rows 0-63 are U = T R, rows 64-127 are P T R = P U.
//   7. O = gamma Q S0^T + P U, scaled, to global (fp32, or bf16 rounded to
//      nearest even when the caller asks for it); U scaled by
//      exp(G_{C-1} - G_r) and written as bf16 hi + lo.
//   8. MMA  U~^T K (or K^T U~) -> TMEM: the state increment.
//   9. S = gamma_{C-1} S + dS in fp32; bf16 hi + lo for step 4.
// Only raw bf16 inputs enter an MMA unsplit; every derived operand (S, Z,
// R, U~) is carried as two bf16 terms so that products keep ~16 mantissa
// bits, and all accumulation is fp32 in TMEM.  Waits on mbarriers are
// bounded; a wait that gives up records GDN_ERR_TIMEOUT in the status word
// and the CTA skips the remaining work and releases its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.h"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {

constexpr int C = 64;            // chunk length (tokens)
constexpr int NT = 256;          // threads per CTA (two warpgroups)
constexpr int FST = 68;          // fp32 row stride of the 64x64 scratch matrices (16-B rows)

// x[j] = TMEM column (col + j) + column (col + off + j), j < N (a multiple of
// 16), of this warp's lane quarter: the hi- and lo-operand halves of a
// product, summed.  16 columns of each half per wait.
template <int N>
__device__ __forceinline__ void tmem_ld_pair(uint32_t col, int off, float (&x)[N]) {
#pragma unroll
    for (int j = 0; j < N; j += 16) {
        float lo[16];
        ptx::tmem_ld16(col + j, *reinterpret_cast<float(*)[16]>(x + j));
        ptx::tmem_ld16(col + off + j, lo);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) x[j + e] += lo[e];
    }
}

// Shared-memory and TMEM map of the state kernel (head_dim 256, and 128 with
// few pairs).  The chunk transform Z = [T; P T] arrives ready-made from the
// workspace (written by chunk_z_kernel), so a CTA only carries BV value rows
// of the state: 64, or 32 to double the CTAs of a small problem.  The tiles
// whose columns are value indices (V, S hi / lo, R / U~ hi / lo) have rows
// of BV bf16: 128 B with the 128-byte swizzle (BV 64), 64 B with the 64-byte
// swizzle (BV 32).
template <int D, int BV_>
struct Cfg {
    static constexpr int BV = BV_;                         // value rows per CTA
    static constexpr int ROWB = 2 * BV;                    // bytes per row of a value tile
    static constexpr uint64_t SWZ = BV == 64 ? ptx::kSwizzle128 : ptx::kSwizzle64;
    static constexpr int NVB = D / BV;                     // CTAs per (sequence, head)
    static constexpr int KT = (D + 127) / 128;            // 128-key tiles of the state update
    static constexpr int NSLAB = D / 64;                   // 64-key slabs of [K;Q]
    static_assert(BV == 64 || BV == 32, "value block of 64 or 32 rows");
    static constexpr int QK_BYTES = NSLAB * 16384;         // one chunk's [K;Q]: NSLAB x (128 rows x 128 B)
    static constexpr int V_BYTES = 64 * ROWB;              // one chunk's V block: 64 rows x ROWB
    static constexpr int ZT_BYTES = 2 * 16384;             // one chunk's Z hi, Z lo: 128 rows x 128 B each
    // PW: a ninth warp issues the loads, into two slots of each streamed tile
    // where shared memory allows, so that the next chunk's tiles land while
    // this one is computed.  Not at head_dim 256 with 64-row blocks: its
    // 64-register state block needs the register budget of eight warps (a
    // ninth rounds the budget to twelve), and only one slot of [K;Q] and V
    // fits.  There one thread per tile (0: [K;Q], 32: V, 64: Z) issues each
    // load as soon as its slot is free.
    static constexpr bool PW = !(D == 256 && BV == 64);
    static constexpr int NQK = PW && D == 128 ? 2 : 1;
    static constexpr int NZS = PW ? 2 : 1;
    static constexpr int NVS = PW ? 2 : 1;
    static constexpr int NTH = PW ? NT + 32 : NT;          // threads per CTA
    // shared memory map (bytes from a 1024-aligned base)
    static constexpr int OFF_QK = 0;
    static constexpr int OFF_V = OFF_QK + NQK * QK_BYTES;
    static constexpr int OFF_Z = OFF_V + NVS * V_BYTES;
    static constexpr int OFF_S = OFF_Z + NZS * ZT_BYTES;   // S hi, S lo: D rows x ROWB each
    static constexpr int OFF_RU = OFF_S + 2 * D * ROWB;    // R (then U~) hi, lo: 64 rows x ROWB
    static constexpr int OFF_MISC = OFF_RU + 2 * 64 * ROWB; // 2 gate sets: G, beta, gamma, end-decay
    static constexpr int OFF_NRM = OFF_MISC + 2 * 4 * 64 * 4;  // 1/|k|, 1/|q| of the chunk
    static constexpr int SMEM = OFF_NRM + 2 * 64 * 4 + 1024;   // + alignment slack
    // A split operand's hi and lo tiles lie one tile apart, so that a single
    // MMA takes both as one B operand of N = 2 BV (its second 64- or 128-byte
    // atom column is the lo tile: LBO = the tile size).  The products then
    // land in two column halves, summed by the epilogue that reads them.
    static constexpr int LBO_S = D * ROWB;                 // S hi -> S lo
    static constexpr int LBO_RU = 64 * ROWB;               // R (U~) hi -> lo
    // TMEM columns: X, Y and each 128-key tile of dS take 2 BV (hi | lo half)
    static constexpr int COL_X = 0;
    static constexpr int COL_Y = 2 * BV;
    static constexpr int COL_DS = 4 * BV;
    static constexpr int TMEM_COLS = COL_DS + 2 * KT * BV <= 256 ? 256 : 512;
    static_assert(COL_DS + 2 * KT * BV <= TMEM_COLS, "TMEM columns");
    static_assert(SMEM + 256 <= 232448, "shared memory (dynamic + static)");
    static_assert(OFF_V % 1024 == 0 && V_BYTES % 1024 == 0 && OFF_Z % 1024 == 0 && OFF_S % 1024 == 0 && OFF_RU % 1024 == 0 &&
                  (D * ROWB) % 1024 == 0 && (64 * ROWB) % 1024 == 0,
                  "swizzled tiles on 1024-byte boundaries");
};

// Bytes of one chunk's Z = [T; P T] in the workspace: bf16 hi then lo, each
// 128 rows x 64 columns in the 128-byte-swizzled layout the MMA reads.
constexpr int Z_BYTES = 2 * 16384;

// Shared-memory map of chunk_z_kernel (head_dim D): [K;Q] for the K K^T /
// Q K^T product, then (reusing the same bytes once that product is done)
// A -> T (fp32), P as bf16 hi / lo tiles, and the Z tile.  The P T product
// reads 128 A rows from P hi: rows 0-63 are P hi, 64-127 are P lo; its third
// term reads 128 rows from P lo, whose rows 64-127 fall on the Z tile (those
// products land in TMEM lanes that are never read).
template <int D>
struct ZCfg {
    static constexpr int SZ_F = 64 * FST * 4;              // one 64 x 64 fp32 matrix
    static constexpr int OFF_QK = 0;                       // D/64 slabs x (K 8 KB | Q 8 KB)
    static constexpr int OFF_A = 0;                        // A, then T in place
    static constexpr int OFF_PHI = 18432;                  // P hi: 64 rows x 128 B (swizzled)
    static constexpr int OFF_PLO = OFF_PHI + 8192;         // P lo
    static constexpr int OFF_Z = OFF_PLO + 8192;           // Z hi | Z lo
    static constexpr int REGION = (D / 64) * 16384 > OFF_Z + Z_BYTES ? (D / 64) * 16384
                                                                     : OFF_Z + Z_BYTES;
    static constexpr int OFF_MISC = REGION;                // G, beta, 1/|k|, 1/|q|
    static constexpr int SMEM = OFF_MISC + 4 * 64 * 4 + 1024;
    static_assert(SZ_F <= OFF_PHI, "A / T below the P tiles");
    static_assert(OFF_PHI % 1024 == 0 && OFF_Z % 1024 == 0, "swizzled tiles on 1024-byte boundaries");
    static_assert(16 * 96 * 4 <= Z_BYTES, "solve scratch inside the Z tile");
};

struct Bars {
    uint64_t tma;
    uint64_t mma;
    uint32_t tmem_base;
    int abort;
};

// Barriers of the state walk: a full / empty pair for each slot of each
// streamed tile ([K;Q], V, Z), the MMA-completion barrier, the TMEM base
// and the abort flag.
struct WalkBars {
    uint64_t full_qk[2], empty_qk[2];
    uint64_t full_v[2], empty_v[2];
    uint64_t full_z[2], empty_z[2];
    uint64_t mma;
    uint32_t tmem_base;
    int abort;
};

// exp(x) via the hardware 2^x; results below the fp32 normal range flush to
// zero (a decay factor under 1e-38 is zero for every purpose here).
__device__ __forceinline__ float fast_exp(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.4426950408889634f));
    return y;
}

// 1 / |x| from a squared norm, 0 for a zero vector (q / k normalisation).
__device__ __forceinline__ float inv_norm(float sq) { return sq > 0.f ? rsqrtf(sq) : 0.f; }

// Squared norms of K row r and Q row r of a stacked [K;Q] stage: NSLAB slabs
// of 64 keys, 16384 bytes apart, each holding 64 K rows then 64 Q rows of
// 128 bytes (128-byte swizzled; a sum of squares does not depend on the order
// in which a row's 16-byte pieces are visited).
template <int NSLAB>
__device__ __forceinline__ void qk_row_sumsq(const uint8_t *qk, int r, float &kk, float &qq) {
    kk = 0.f;
    qq = 0.f;
#pragma unroll
    for (int sl = 0; sl < NSLAB; ++sl) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 a = *reinterpret_cast<const uint4 *>(qk + sl * 16384 + r * 128 + c * 16);
            const uint4 b =
                *reinterpret_cast<const uint4 *>(qk + sl * 16384 + 8192 + r * 128 + c * 16);
            const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float k0 = __uint_as_float(wa[e] << 16), k1 = __uint_as_float(wa[e] & 0xffff0000u);
                const float q0 = __uint_as_float(wb[e] << 16), q1 = __uint_as_float(wb[e] & 0xffff0000u);
                kk = fmaf(k0, k0, fmaf(k1, k1, kk));
                qq = fmaf(q0, q0, fmaf(q1, q1, qq));
            }
        }
    }
}

// Store 16 consecutive fp32 values as bf16 hi / lo into two 128-B-swizzled
// tiles at (row, col0 .. col0+15); col0 is a multiple of 8.  hi keeps the top
// 16 bits of each value, lo = bf16_rn(x - hi): ~16 significant bits together.
template <int ROWB = 128>
__device__ __forceinline__ void store_split16(uint8_t *hi_tile, uint8_t *lo_tile, int row, int col0,
                                              const float (&x)[16]) {
    ptx::store_split8<ROWB>(hi_tile, lo_tile, row, col0, *reinterpret_cast<const float(*)[8]>(x));
    ptx::store_split8<ROWB>(hi_tile, lo_tile, row, col0 + 8,
                            *reinterpret_cast<const float(*)[8]>(x + 8));
}

// Warp-level bf16 MMA, m16n8k16, fp32 accumulate in place: d += a b.
// Fragments (lane = 4 g + c): a0 = A[g][2c..2c+1], a1 = A[g+8][2c..2c+1],
// a2 = A[g][2c+8..2c+9], a3 = A[g+8][2c+8..2c+9]; b0 = B[2c..2c+1][g],
// b1 = B[2c+8..2c+9][g]; d0, d1 = D[g][2c..2c+1], d2, d3 = D[g+8][2c..2c+1];
// the element with the lower index in the low half of each 32-bit word.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// A fragment of the 16 x 16 fp32 block at `base` (row stride ld), as bf16
// hi / lo words (~16 significant bits together).
__device__ __forceinline__ void frag_a(const float *base, int ld, int lane, uint32_t (&hi)[4],
                                       uint32_t (&lo)[4]) {
    const int g = lane >> 2, c = lane & 3;
    const float2 v0 = *reinterpret_cast<const float2 *>(base + g * ld + 2 * c);
    const float2 v1 = *reinterpret_cast<const float2 *>(base + (g + 8) * ld + 2 * c);
    const float2 v2 = *reinterpret_cast<const float2 *>(base + g * ld + 2 * c + 8);
    const float2 v3 = *reinterpret_cast<const float2 *>(base + (g + 8) * ld + 2 * c + 8);
    ptx::split_pair(v0.x, v0.y, hi[0], lo[0]);
    ptx::split_pair(v1.x, v1.y, hi[1], lo[1]);
    ptx::split_pair(v2.x, v2.y, hi[2], lo[2]);
    ptx::split_pair(v3.x, v3.y, hi[3], lo[3]);
}

// B fragment of the 16 x 8 fp32 block at `base` (B[k][n] at base[k * ld + n]).
__device__ __forceinline__ void frag_b(const float *base, int ld, int lane, uint32_t (&hi)[2],
                                       uint32_t (&lo)[2]) {
    const int g = lane >> 2, c = lane & 3;
    const float x0 = base[(2 * c) * ld + g], x1 = base[(2 * c + 1) * ld + g];
    const float x2 = base[(2 * c + 8) * ld + g], x3 = base[(2 * c + 9) * ld + g];
    ptx::split_pair(x0, x1, hi[0], lo[0]);
    ptx::split_pair(x2, x3, hi[1], lo[1]);
}

// d += A B for split operands: A hi B hi + A hi B lo + A lo B hi.
__device__ __forceinline__ void mma3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                     const uint32_t (&bh)[2], const uint32_t (&bl)[2]) {
    mma16816(d, ah, bh);
    mma16816(d, ah, bl);
    mma16816(d, al, bh);
}

// T = (I + A)^-1 for a strictly lower triangular 64x64 A stored in full
// (zeros on and above the diagonal, row stride FST), in place, on 256
// threads t = 0..255 (8 warps) sharing hardware barrier `bar`, with two
// 32x32 diagonal blocks:
//   1. T_00 = (I + A_00)^-1 and T_11 = (I + A_11)^-1 by column substitution
//      on CUDA cores, one column per thread (warp 1: block 0, warp 3:
//      block 1, on SMSPs 1 and 3 of the stream's warps 8-15, away from the
//      threads that issue products and copies; every lane of a warp reads
//      the same row of A, a broadcast)
//   2. X = T_11 A_10 (32x32, into W): eight 16 x 8 tiles, warp-level MMAs
//   3. T_10 = -X T_00: eight tiles, warp-level MMAs
// which is block forward substitution: A_10 T_00 + (I + A_11) T_10 = 0.
// The products are 16-row blocks, too small for a 128-row tensor-memory
// MMA, so the warps use register-operand MMAs on bf16 hi / lo splits (three
// terms, ~16 significant bits, fp32 accumulation).  The result is T in full
// (zeros above the diagonal); entered and left with the matrix visible to
// all participants.
__device__ __forceinline__ void ut_transform32(float *sAT, float *sW, int t, int bar) {
    constexpr int LW = 40;                            // row stride of W (32 x 32 fp32)
    const int warp = t >> 5, lane = t & 31;
    const int g = lane >> 2, c = lane & 3;
    // 1. diagonal blocks: x = column j of T_bb, x[r] = -sum_{i<r} A[r][i] x[i]
    //    below the diagonal (four partial sums per row)
    float x[32];
    const bool subst = (warp == 1 || warp == 3);
    const int blk = (warp == 3) ? 1 : 0, j = lane;
    if (subst) {
        const float *Ab = sAT + (blk * 32) * FST + blk * 32;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i4 = 0; i4 < 32; i4 += 4) {
                if (i4 < r) {
                    const float4 a = *reinterpret_cast<const float4 *>(Ab + r * FST + i4);
                    acc[0] = fmaf(a.x, x[i4], acc[0]);
                    if (i4 + 1 < r) acc[1] = fmaf(a.y, x[i4 + 1], acc[1]);
                    if (i4 + 2 < r) acc[2] = fmaf(a.z, x[i4 + 2], acc[2]);
                    if (i4 + 3 < r) acc[3] = fmaf(a.w, x[i4 + 3], acc[3]);
                }
            }
            const float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            x[r] = (r == j) ? 1.f : ((r > j) ? -sum : 0.f);
        }
    }
    ptx::named_sync(bar, 256);
    if (subst) {
        float *Tb = sAT + (blk * 32) * FST + blk * 32;
#pragma unroll
        for (int r = 0; r < 32; ++r) Tb[r * FST + j] = x[r];
    }
    ptx::named_sync(bar, 256);
    // 2. X = T_11 A_10: warp -> rows 16 m0 .. +15, columns 8 n0 .. +7
    const int m0 = (warp >> 2) * 16, n0 = (warp & 3) * 8;
    {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 32; ks += 16) {
            uint32_t ah[4], al[4], bh[2], bl[2];
            frag_a(sAT + (32 + m0) * FST + 32 + ks, FST, lane, ah, al);    // T_11 rows, k block
            frag_b(sAT + (32 + ks) * FST + n0, FST, lane, bh, bl);         // A_10 k rows, n cols
            mma3(d, ah, al, bh, bl);
        }
        float *w = sW + m0 * LW + n0 + 2 * c;
        *reinterpret_cast<float2 *>(w + g * LW) = make_float2(d[0], d[1]);
        *reinterpret_cast<float2 *>(w + (g + 8) * LW) = make_float2(d[2], d[3]);
    }
    ptx::named_sync(bar, 256);
    // 3. T_10 = -X T_00 over A_10's place
    {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 32; ks += 16) {
            uint32_t ah[4], al[4], bh[2], bl[2];
            frag_a(sW + m0 * LW + ks, LW, lane, ah, al);                   // X rows, k block
            frag_b(sAT + ks * FST + n0, FST, lane, bh, bl);                // T_00 k rows, n cols
            mma3(d, ah, al, bh, bl);
        }
        float *o = sAT + (32 + m0) * FST + n0 + 2 * c;
        *reinterpret_cast<float2 *>(o + g * FST) = make_float2(-d[0], -d[1]);
        *reinterpret_cast<float2 *>(o + (g + 8) * FST) = make_float2(-d[2], -d[3]);
    }
    ptx::named_sync(bar, 256);
}

// The same T = (I + A)^-1 with the off-diagonal block in one round of
// register-resident MMAs.  Threads t = 0..255 of one stream share hardware
// barrier `bar`; threads 0-127 also share `bar4`:
//   1. T_00 and T_11 by column substitution (as in ut_transform32) on warps 1
//      and 3 of the stream, which sit on the SMSPs of no issuing thread (a
//      warp blocked issuing a product or a copy holds back the other warps
//      of its SMSP)
//   2. T_10 = -(T_11 A_10) T_00 by warps 0-3: warp w forms the 16-row band
//      16 (w >> 1) of X = T_11 A_10 (all 32 columns; the two warps of a band
//      compute it twice) and feeds its accumulators straight back as the A
//      operand of the product with T_00, for 16 output columns 16 (w & 1).
//      k blocks that meet only the zero triangle of T_11 or T_00 are skipped.
// One round and two barriers instead of X through shared memory.  Same
// operands and result as ut_transform32.  Used by chunk_z_kernel, where
// three CTAs share an SM (8 x 16384 x 16 x 256: 4.65 -> 4.59 ms); in
// chunked_d128_kernel, whose state stream shares the SMSPs, ut_transform32
// measured faster.
__device__ __forceinline__ void ut_transform32r(float *sAT, int t, int bar, int bar4) {
    const int warp = t >> 5, lane = t & 31;
    if ((warp == 1 || warp == 3)) {
        const int blk = warp >> 1, j = lane;
        float *Ab = sAT + (blk * 32) * FST + blk * 32;
        float x[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i4 = 0; i4 < 32; i4 += 4) {
                if (i4 < r) {
                    const float4 a = *reinterpret_cast<const float4 *>(Ab + r * FST + i4);
                    acc[0] = fmaf(a.x, x[i4], acc[0]);
                    if (i4 + 1 < r) acc[1] = fmaf(a.y, x[i4 + 1], acc[1]);
                    if (i4 + 2 < r) acc[2] = fmaf(a.z, x[i4 + 2], acc[2]);
                    if (i4 + 3 < r) acc[3] = fmaf(a.w, x[i4 + 3], acc[3]);
                }
            }
            const float sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            x[r] = (r == j) ? 1.f : ((r > j) ? -sum : 0.f);
        }
        __syncwarp();                                 // every lane has read A_bb
#pragma unroll
        for (int r = 0; r < 32; ++r) Ab[r * FST + j] = x[r];
    }
    ptx::named_sync(bar, 256);
    if (t < 128) {
        const int g = lane >> 2, c = lane & 3;
        const int mb = warp >> 1, nh = warp & 1;
        // X band: rows 16 mb .. +15 of T_11 A_10 (row m of T_11 is zero past column m)
        float d[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 32; ks += 16) {
            if (mb == 0 && ks == 16) continue;
            uint32_t ah[4], al[4];
            frag_a(sAT + (32 + 16 * mb) * FST + 32 + ks, FST, lane, ah, al);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                uint32_t bh[2], bl[2];
                frag_b(sAT + (32 + ks) * FST + 8 * nt, FST, lane, bh, bl);
                mma3(d[nt], ah, al, bh, bl);
            }
        }
        // columns 16 nh .. +15 of -X T_00 (rows 0-15 of T_00 are zero past column 15)
        float e[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) e[nt][0] = e[nt][1] = e[nt][2] = e[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 32; ks += 16) {
            if (nh == 1 && ks == 0) continue;
            const int t0 = ks / 8, t1 = t0 + 1;
            uint32_t ah[4], al[4];
            ptx::split_pair(d[t0][0], d[t0][1], ah[0], al[0]);
            ptx::split_pair(d[t0][2], d[t0][3], ah[1], al[1]);
            ptx::split_pair(d[t1][0], d[t1][1], ah[2], al[2]);
            ptx::split_pair(d[t1][2], d[t1][3], ah[3], al[3]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                uint32_t bh[2], bl[2];
                frag_b(sAT + ks * FST + 16 * nh + 8 * nt, FST, lane, bh, bl);
                mma3(e[nt], ah, al, bh, bl);
            }
        }
        ptx::named_sync(bar4, 128);                   // every band has read A_10
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float *o = sAT + (32 + 16 * mb) * FST + 16 * nh + 8 * nt + 2 * c;
            *reinterpret_cast<float2 *>(o + g * FST) = make_float2(-e[nt][0], -e[nt][1]);
            *reinterpret_cast<float2 *>(o + (g + 8) * FST) = make_float2(-e[nt][2], -e[nt][3]);
        }
    }
    ptx::named_sync(bar, 256);
}

// The same T = (I + A)^-1 with four 16x16 diagonal blocks: shorter
// column substitutions, two more rounds of MMAs.  Same operands, threads and
// result as ut_transform32:
//   1. T_ii = (I + A_ii)^-1 for the four diagonal blocks (column
//      substitution on CUDA cores, one column per thread)
//   2. X_i = T_ii A[i, :i] for i = 1..3, all at once (into W, 16 x 96 fp32):
//      twelve 16 x 8 tiles, warp-level MMAs
//   3. T[i, :i] = -X_i T[:i, :i] for i = 1, 2, 3 in turn (2i tiles each)
// which is block forward substitution: (I + A)_ii T_ij + sum_k A_ik T_kj = 0.
// Measured faster than ut_transform32 where the transform stream limits the
// chunk (head_dim 64), slower at head_dim 128.
__device__ __forceinline__ void ut_transform16(float *sAT, float *sW, int t, int bar) {
    constexpr int LW = 96;                            // row stride of W
    const int warp = t >> 5, lane = t & 31;
    const int g = lane >> 2, c = lane & 3;
    // 1. diagonal blocks
    float x[16];
    const int blk = t >> 4, j = t & 15;
    if (t < 64) {
        const float *Ab = sAT + (blk * 16) * FST + blk * 16;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float a[16];
#pragma unroll
            for (int i4 = 0; i4 < 16; i4 += 4) {
                if (i4 < r) {
                    const float4 v = *reinterpret_cast<const float4 *>(Ab + r * FST + i4);
                    a[i4] = v.x; a[i4 + 1] = v.y; a[i4 + 2] = v.z; a[i4 + 3] = v.w;
                }
            }
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) acc = fmaf(a[i], x[i], acc);
            x[r] = (r == j) ? 1.f : ((r > j) ? -acc : 0.f);
        }
    }
    ptx::named_sync(bar, 256);
    if (t < 64) {
        float *Tb = sAT + (blk * 16) * FST + blk * 16;
#pragma unroll
        for (int r = 0; r < 16; ++r) Tb[r * FST + j] = x[r];
    }
    ptx::named_sync(bar, 256);
    // 2. X_i = T_ii A[i, :i]: tile q (12 of them) -> block row i, columns n0 .. n0+7
    for (int q = warp; q < 12; q += 8) {
        const int i = q < 2 ? 1 : (q < 6 ? 2 : 3);
        const int n0 = 8 * (q - (i == 1 ? 0 : (i == 2 ? 2 : 6)));
        uint32_t ah[4], al[4], bh[2], bl[2];
        frag_a(sAT + (16 * i) * FST + 16 * i, FST, lane, ah, al);      // T_ii
        frag_b(sAT + (16 * i) * FST + n0, FST, lane, bh, bl);           // A[i, n0 ..]
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma3(d, ah, al, bh, bl);
        float *w = sW + 8 * (i - 1) * i + n0 + 2 * c;                   // X_i at column 16 (i-1) i / 2
        *reinterpret_cast<float2 *>(w + g * LW) = make_float2(d[0], d[1]);
        *reinterpret_cast<float2 *>(w + (g + 8) * LW) = make_float2(d[2], d[3]);
    }
    ptx::named_sync(bar, 256);
    // 3. block rows in turn (each needs the rows above it): T[i, n0 .. n0+7]
    //    = -sum over 16-wide k blocks of X_i[:, k] T[k, n0 ..]
#pragma unroll
    for (int i = 1; i <= 3; ++i) {
        if (warp < 2 * i) {
            const int n0 = 8 * warp;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            for (int ks = 0; ks < i; ++ks) {
                uint32_t ah[4], al[4], bh[2], bl[2];
                frag_a(sW + 8 * (i - 1) * i + 16 * ks, LW, lane, ah, al);   // X_i, k block ks
                frag_b(sAT + (16 * ks) * FST + n0, FST, lane, bh, bl);     // T[ks block, n0 ..]
                mma3(d, ah, al, bh, bl);
            }
            float *o = sAT + (16 * i) * FST + n0 + 2 * c;
            *reinterpret_cast<float2 *>(o + g * FST) = make_float2(-d[0], -d[1]);
            *reinterpret_cast<float2 *>(o + (g + 8) * FST) = make_float2(-d[2], -d[3]);
        }
        ptx::named_sync(bar, 256);
    }
}

// ---------------------------------------------------------------------------
// Chunk transform for head_dim 256, and for head_dim 128 with few (sequence,
// head) pairs: Z = [T; P T] of every (sequence, head, chunk), independent of
// the state, computed once per chunk (not once per value block) into the
// workspace.  Persistent CTAs walk the chunks:
//   1. TMA brings K and Q (stacked per 64-key slab), plain loads the gates;
//   2. MMA [K;Q] K^T -> TMEM (M = 128, N = 64, K = D): K K^T and Q K^T;
//   3. A and P, T = (I + A)^-1 by 32 x 32 blocks, MMA [P hi; P lo] T, and
//      Z = [T; P T] as bf16 hi + lo in the swizzled tile layout;
//   4. one bulk copy writes the 32 KB tile to the workspace.
template <int D, bool NORM>
__global__ void __launch_bounds__(NT, 3)
chunk_z_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const float *__restrict__ g, const float *__restrict__ beta,
               uint8_t *__restrict__ zws, int T, int H, int Hk, int n_chunks, int n_tasks,
               int *status)
{
    using ZC = ZCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ Bars bars;
    float *sG = reinterpret_cast<float *>(sm + ZC::OFF_MISC);
    float *sBeta = sG + 64;
    float *sNk = sG + 128, *sNq = sG + 192;          // with q / k normalisation
    uint8_t *sQK = sm + ZC::OFF_QK;
    float *sA = reinterpret_cast<float *>(sm + ZC::OFF_A);
    uint8_t *sPhi = sm + ZC::OFF_PHI, *sPlo = sm + ZC::OFF_PLO;
    uint8_t *sZhi = sm + ZC::OFF_Z, *sZlo = sm + ZC::OFF_Z + 16384;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int wg = tid >> 7;
    const int row = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // The state walk that follows may be scheduled as soon as every CTA of
    // this grid has started: it reads the workspace only after its grid
    // dependency wait, which returns once this grid has completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (tid == 0) {
        bars.abort = 0;
        ptx::mbar_init(&bars.tma, 1);
        ptx::mbar_init(&bars.mma, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
    }
    if (warp == 0) {
        ptx::tmem_alloc(&bars.tmem_base, 64);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    volatile int *abort_flag = &bars.abort;
    auto fail = [&]() {
        if (atomicExch(const_cast<int *>(abort_flag), 1) == 0) atomicExch(status, GDN_ERR_TIMEOUT);
    };
    const uint32_t aQK = ptx::smem_u32(sQK);

    uint32_t phase = 0, mma_phase = 0;                // TMA and MMA barrier phases
    bool tma_pending = false;                         // thread 0: a load not yet waited for
    // A task's [K;Q] tile and gates are fetched during the task before it:
    // the gates (threads 0-63, into registers) once that task's P T product
    // has completed, and the tile at the same point where its bytes no longer
    // overlap anything live (head_dim 64 and 128: the tile ends below the Z
    // tile; at 256 it covers Z and is fetched once Z has been stored).
    constexpr bool kTileEarly = (D / 64) * 16384 <= ZC::OFF_Z;
    auto issue_tile = [&](int tsk) {                  // thread 0
        const int cc = tsk % n_chunks, bbh = tsk / n_chunks;
        const int bb = bbh / H, hh = bbh - bb * H;
        constexpr uint32_t bytes = (uint32_t)(D / 64) * 2 * 8192;
        ptx::mbar_arrive_expect_tx(&bars.tma, bytes);
        tma_pending = true;
#pragma unroll
        for (int sl = 0; sl < D / 64; ++sl) {
            ptx::tma_load_4d(sQK + sl * 16384, &tm_k, &bars.tma, sl * 64, hh % Hk, cc * C, bb);
            ptx::tma_load_4d(sQK + sl * 16384 + 8192, &tm_q, &bars.tma, sl * 64, hh % Hk, cc * C,
                             bb);
        }
    };
    float gnext = 0.f, bnext = 0.f;                   // threads 0-63: the next task's gates
    auto load_gates = [&](int tsk) {
        const int cc = tsk % n_chunks, bbh = tsk / n_chunks;
        const int bb = bbh / H, hh = bbh - bb * H;
        gnext = 0.f;
        bnext = 0.f;
        if (tid < min(C, T - cc * C)) {
            const size_t gi = ((size_t)bb * T + cc * C + tid) * H + hh;
            gnext = g[gi];
            bnext = beta[gi];
        }
    };
    if (blockIdx.x < n_tasks) {
        if (tid == 0) issue_tile(blockIdx.x);
        if (tid < 64) load_gates(blockIdx.x);
    }
    for (int task = blockIdx.x; task < n_tasks && !*abort_flag; task += gridDim.x) {
        const int next = task + (int)gridDim.x;

        // 1. this task's gates (fetched during the task before) -> cumsum
        if (tid < 64) {
            const float gr = fmaxf(gnext, -30.f);     // exp(-30) ~ 1e-13: a reset stays a reset
            const float br = bnext;
            const int r = tid;
            float sacc = gr;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, sacc, o);
                if (lane >= o) sacc += y;
            }
            sG[r] = sacc;
            sBeta[r] = br;
        }
        __syncthreads();
        if (tid >= 32 && tid < 64) sG[tid] += sG[31];
        if (!ptx::mbar_wait(&bars.tma, phase, abort_flag)) fail();
        else if (tid == 0) tma_pending = false;
        if constexpr (NORM) {
            if (tid < 64 && !*abort_flag) {
                float kk, qq;
                qk_row_sumsq<D / 64>(sQK, tid, kk, qq);
                sNk[tid] = inv_norm(kk);
                sNq[tid] = inv_norm(qq);
            }
        }
        __syncthreads();
        if (*abort_flag) break;

        // 2. MMA: [K;Q] K^T  (M = 128, N = 64, K = D)
        if (tid == 0) {
            ptx::tc_fence_after();
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 64, false, false);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t a = aQK + (kk >> 2) * 16384 + (kk & 3) * 32;
                const uint64_t da = ptx::smem_desc(a, 16, 1024);
                ptx::mma_bf16(tmem, da, da, idesc, kk > 0);
            }
            ptx::mma_commit(&bars.mma);
        }
        if (!ptx::mbar_wait(&bars.mma, mma_phase, abort_flag)) fail();
        ptx::tc_fence_after();
        phase ^= 1;
        mma_phase ^= 1;

        // 3. A, P (the [K;Q] bytes are free now: the product has completed)
        {
            float kq[32];
            ptx::tmem_ld16(tmem + lane_off + wg * 32, *reinterpret_cast<float(*)[16]>(kq));
            ptx::tmem_ld16(tmem + lane_off + wg * 32 + 16, *reinterpret_cast<float(*)[16]>(kq + 16));
            ptx::tmem_ld_wait();
            const int r = row & 63;
            const float Gr = sG[r];
            // with q / k normalisation A[r,i] and P[r,i] carry nk_i and nk_r / nq_r
            if (row < 64) {
                const float br = NORM ? sBeta[r] * sNk[r] : sBeta[r];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int i = wg * 32 + j;
                    const float kn = NORM ? kq[j] * sNk[i] : kq[j];
                    sA[r * FST + i] = (i < r) ? br * fast_exp(Gr - sG[i]) * kn : 0.f;
                }
            } else {
                const float pr = NORM ? sNq[r] : 1.f;
                float pv[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int i = wg * 32 + j;
                    const float kn = NORM ? kq[j] * sNk[i] : kq[j];
                    pv[j] = (i <= r) ? pr * fast_exp(Gr - sG[i]) * kn : 0.f;
                }
                store_split16(sPhi, sPlo, r, wg * 32, *reinterpret_cast<float(*)[16]>(pv));
                store_split16(sPhi, sPlo, r, wg * 32 + 16, *reinterpret_cast<float(*)[16]>(pv + 16));
            }
        }
        ptx::tc_fence_before();
        __syncthreads();
        ut_transform32r(sA, tid, 0, 1);               // T in place over A
        {                                             // T as hi / lo into Z rows 0-63
            const int r = tid >> 2, c0 = (tid & 3) * 16;
            float t[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) t[e] = sA[r * FST + c0 + e];
            store_split16(sZhi, sZlo, r, c0, t);
        }
        ptx::fence_proxy_async_smem();
        __syncthreads();
        // P T on the tensor cores: A = [P hi; P lo] (128 rows), B = T rows
        // (MN-major), three terms P hi T hi + P hi T lo + P lo T hi summed in
        // TMEM lanes 0-63
        if (tid == 0) {
            ptx::tc_fence_after();
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 64, false, true);
            const uint32_t aP[3] = {ptx::smem_u32(sPhi), ptx::smem_u32(sPhi), ptx::smem_u32(sPlo)};
            const uint32_t bT[3] = {ptx::smem_u32(sZhi), ptx::smem_u32(sZlo), ptx::smem_u32(sZhi)};
#pragma unroll
            for (int part = 0; part < 3; ++part)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    ptx::mma_bf16(tmem, ptx::smem_desc(aP[part] + kk * 32, 16, 1024),
                                  ptx::smem_desc(bT[part] + kk * 2048, 8192, 1024), idesc,
                                  part > 0 || kk > 0);
            ptx::mma_commit(&bars.mma);
        }
        if (!ptx::mbar_wait(&bars.mma, mma_phase, abort_flag)) fail();
        ptx::tc_fence_after();
        mma_phase ^= 1;
        if (next < n_tasks) {                         // the next task's inputs, in flight meanwhile
            if (kTileEarly && tid == 0) issue_tile(next);
            if (tid < 64) load_gates(next);
        }
        if ((warp & 3) < 2) {                         // P T rows -> Z rows 64-127
            float pt[32];
            ptx::tmem_ld16(tmem + lane_off + wg * 32, *reinterpret_cast<float(*)[16]>(pt));
            ptx::tmem_ld16(tmem + lane_off + wg * 32 + 16, *reinterpret_cast<float(*)[16]>(pt + 16));
            ptx::tmem_ld_wait();
            store_split16(sZhi, sZlo, 64 + row, wg * 32, *reinterpret_cast<float(*)[16]>(pt));
            store_split16(sZhi, sZlo, 64 + row, wg * 32 + 16, *reinterpret_cast<float(*)[16]>(pt + 16));
        }
        // 4. the tile to the workspace (one bulk copy), then the buffer is free
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            ptx::bulk_store(zws + (size_t)task * Z_BYTES, sZhi, Z_BYTES);
            ptx::bulk_commit_group();
            ptx::bulk_wait_read_all();
            if (!kTileEarly && next < n_tasks) issue_tile(next);   // Z has left the tile's bytes
        }
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
    }
    if (tid == 0) {
        ptx::bulk_wait_all();
        if (tma_pending) {                            // after an abort: let the load land
            const volatile int never = 0;
            ptx::mbar_wait(&bars.tma, phase, &never, 1000000000LL);
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, 64);
}

template <int D, int BV_, bool NORM>
__global__ void __launch_bounds__(Cfg<D, BV_>::NTH, 1)
chunked_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const float *__restrict__ g,
               const float *__restrict__ beta, const float *state_in, float *state_out,
               float *__restrict__ out, const uint8_t *__restrict__ zws, int T, int H, int Hk,
               float scale, int *status, bool out_bf16, int pair0)
{
    using CF = Cfg<D, BV_>;
    constexpr int BV = CF::BV;
    constexpr int ROWB = CF::ROWB;
    constexpr int KT = CF::KT;
    constexpr int HALF = BV / 2;          // value columns per warpgroup
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ WalkBars bars;
    float *gsets = reinterpret_cast<float *>(sm + CF::OFF_MISC);   // set i: gsets + 256 i
    float *sNk = reinterpret_cast<float *>(sm + CF::OFF_NRM), *sNq = sNk + 64;
    uint8_t *sQK0 = sm + CF::OFF_QK;      // slot s at + s * QK_BYTES
    uint8_t *sV0 = sm + CF::OFF_V;        // slot s at + s * V_BYTES
    uint8_t *sZ0 = sm + CF::OFF_Z;        // slot s at + s * Z_BYTES (hi, then lo)
    uint8_t *sShi = sm + CF::OFF_S, *sSlo = sm + CF::OFF_S + D * ROWB;
    uint8_t *sRhi = sm + CF::OFF_RU, *sRlo = sm + CF::OFF_RU + 64 * ROWB;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int wg = tid >> 7;                 // warpgroup: which half of the value columns
    const int row = tid & 127;               // TMEM lane this thread reads
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    constexpr bool PW = CF::PW;
    const bool producer = PW && warp == NT / 32;   // warp 8: the loads; warps 0-7: the chain
    // the value blocks of one head are neighbours in the grid, so they share
    // their [K;Q] and Z reads through L2
    const int bh = pair0 + (int)(blockIdx.x / CF::NVB);   // (sequence, head) pair
    const int b = bh / H, h = bh - b * H;
    const int v0 = (blockIdx.x % CF::NVB) * BV;
    const int n_chunks = (T + C - 1) / C;
    const uint8_t *zbh = zws + (size_t)bh * n_chunks * Z_BYTES;

    if (tid == 0) {
        bars.abort = 0;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&bars.full_qk[s], 1);
            ptx::mbar_init(&bars.empty_qk[s], 1);
            ptx::mbar_init(&bars.full_v[s], 1);
            ptx::mbar_init(&bars.empty_v[s], 1);
            ptx::mbar_init(&bars.full_z[s], 1);
            ptx::mbar_init(&bars.empty_z[s], 1);
        }
        ptx::mbar_init(&bars.mma, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 0) {
        ptx::tmem_alloc(&bars.tmem_base, CF::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // ---- initial state block into registers (warps 0-7): key = kt*128 +
    //      row, values v0 + wg*HALF + j; coalesced over keys
    float S[KT][HALF];
    const size_t st_base = (size_t)bh * D * D;
    if (!producer) {
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
            const int key = kt * 128 + row;
#pragma unroll
            for (int j = 0; j < HALF; ++j) {
                const int v = v0 + wg * HALF + j;
                S[kt][j] = (state_in && key < D) ? state_in[st_base + (size_t)v * D + key] : 0.f;
            }
        }
        // S hi / lo tiles: row = key, columns = value index within the block
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
            const int key = kt * 128 + row;
            if (key < D) {
#pragma unroll
                for (int j = 0; j < HALF; j += 16) {
                    float x[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = S[kt][j + e];
                    store_split16<ROWB>(sShi, sSlo, key, wg * HALF + j, x);
                }
            }
        }
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    volatile int *abort_flag = &bars.abort;
    auto fail = [&]() {
        if (atomicExch(const_cast<int *>(abort_flag), 1) == 0) atomicExch(status, GDN_ERR_TIMEOUT);
    };

    // ---- loads (lane 0 of warp 8; without it threads 0, 32 and 64, one per
    // tile).  Chunk c's [K;Q], V and Z go to slot c % (slots of that tile);
    // the issuing thread records the last chunk it loaded into each slot.
    int last_qk[2] = {-1, -1}, last_v[2] = {-1, -1}, last_z[2] = {-1, -1};
    auto issue_v = [&](int c) {
        const int sv = c % CF::NVS;
        ptx::mbar_arrive_expect_tx(&bars.full_v[sv], CF::V_BYTES);
        ptx::tma_load_4d(sV0 + sv * CF::V_BYTES, &tm_v, &bars.full_v[sv], v0, h, c * C, b);
        last_v[sv] = c;
    };
    // Z as eight 4 KB copies: one 32 KB bulk copy was measured to land more
    // than a chunk step after it was issued, several smaller ones in flight
    // at once land sooner.
    auto issue_z = [&](int c) {
        const int sz = c % CF::NZS;
        ptx::mbar_arrive_expect_tx(&bars.full_z[sz], Z_BYTES);
#pragma unroll
        for (int part = 0; part < 8; ++part)
            ptx::bulk_load(sZ0 + sz * Z_BYTES + part * (Z_BYTES / 8),
                           zbh + (size_t)c * Z_BYTES + part * (Z_BYTES / 8), Z_BYTES / 8,
                           &bars.full_z[sz]);
        last_z[sz] = c;
    };
    auto issue_qk = [&](int c) {
        const int sq = c % CF::NQK;
        ptx::mbar_arrive_expect_tx(&bars.full_qk[sq], CF::QK_BYTES);
        uint8_t *dst = sQK0 + sq * CF::QK_BYTES;
#pragma unroll
        for (int s = 0; s < D / 64; ++s) {
            ptx::tma_load_4d(dst + s * 16384, &tm_k, &bars.full_qk[sq], s * 64, h % Hk, c * C, b);
            ptx::tma_load_4d(dst + s * 16384 + 8192, &tm_q, &bars.full_qk[sq], s * 64, h % Hk,
                             c * C, b);
        }
        last_qk[sq] = c;
    };
    // every copy addressed to this CTA's shared memory lands before the CTA
    // can exit (a bounded wait; on the normal path each of these phases has
    // completed already)
    auto drain = [&]() {
        const volatile int never = 0;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            if (last_v[s] >= 0)
                ptx::mbar_wait(&bars.full_v[s], (uint32_t)((last_v[s] / CF::NVS) & 1), &never,
                               1000000000LL);
            if (last_z[s] >= 0)
                ptx::mbar_wait(&bars.full_z[s], (uint32_t)((last_z[s] / CF::NZS) & 1), &never,
                               1000000000LL);
            if (last_qk[s] >= 0)
                ptx::mbar_wait(&bars.full_qk[s], (uint32_t)((last_qk[s] / CF::NQK) & 1), &never,
                               1000000000LL);
        }
    };

    if (producer) {
        // Warp 8 refills a slot once the chunk that used it before has
        // released it: V after its R epilogue, Z and [K;Q] when the last
        // product reading them completes.  With two slots the loads run one
        // chunk ahead of the products.  The order V, Z, [K;Q] is the order in
        // which a chunk releases them.  A wait that gives up here records
        // the timeout in the status word only: the abort flag is written by
        // warps 0-7 alone, always before a barrier they all pass, so that
        // they all read the same value after it; they then give up on their
        // own bounded waits for the loads that never come.
        if (lane == 0) {
            int c = 0;
            for (; c < n_chunks; ++c) {
                const int sq = c % CF::NQK, sv = c % CF::NVS, sz = c % CF::NZS;
                if (c == 0) {
                    // chunk 0: its V and [K;Q] come from the caller's inputs;
                    // Z is the transform kernel's output, read only once that
                    // grid has completed (this grid may start before, as a
                    // programmatic dependent launch)
                    issue_v(0);
                    issue_qk(0);
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                    issue_z(0);
                    continue;
                }
                if (c >= CF::NVS && !ptx::mbar_wait(&bars.empty_v[sv],
                                                    (uint32_t)((c / CF::NVS - 1) & 1), abort_flag))
                    break;
                issue_v(c);
                if (c >= CF::NZS && !ptx::mbar_wait(&bars.empty_z[sz],
                                                    (uint32_t)((c / CF::NZS - 1) & 1), abort_flag))
                    break;
                issue_z(c);
                if (c >= CF::NQK && !ptx::mbar_wait(&bars.empty_qk[sq],
                                                    (uint32_t)((c / CF::NQK - 1) & 1), abort_flag))
                    break;
                issue_qk(c);
            }
            if (c < n_chunks && !*abort_flag)
                atomicExch(status, GDN_ERR_TIMEOUT);   // gave up with loads still to issue
            drain();
        }
        __syncwarp();
    } else {
        uint32_t mma_phase = 0;
        // wait for the next MMA commit (warps 0-7)
        auto wait_mma = [&]() {
            if (!ptx::mbar_wait(&bars.mma, mma_phase, abort_flag)) fail();
            mma_phase ^= 1;
            ptx::tc_fence_after();
        };
        const size_t tok_stride = (size_t)H * D;

        // Gates: warps 2 and 3 (threads 64-127, TMEM lanes 64-127, idle while
        // the other warps build R) scan the next chunk's g into the other of
        // two gate sets during step 5, from g and beta they loaded one chunk
        // earlier; the set of chunk 0 is built here.  Set layout: G (in-chunk
        // running sum of g, each clamped at -30: exp(-30) ~ 1e-13, a reset
        // stays a reset), beta, gamma = exp(G), end-decay = exp(G_63 - G).
        const bool gate_thread = tid >= 64 && tid < 128;
        const int gr_ = tid - 64;                      // token of the chunk (gate threads)
        float gnext = 0.f, bnext = 0.f;
        // g, beta of chunk cc into gnext / bnext.  Nothing reads them until
        // the scan a chunk later, so the loads stay in flight meanwhile.
        auto load_gates = [&](int cc) {
            gnext = 0.f;
            bnext = 0.f;
            if (cc * C + gr_ < T) {
                const size_t gi = ((size_t)b * T + cc * C + gr_) * H + h;
                gnext = g[gi];
                bnext = beta[gi];
            }
        };
        auto scan_gates = [&](float *set) {           // gate threads only
            float sacc = fmaxf(gnext, -30.f);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, sacc, o);
                if (lane >= o) sacc += y;
            }
            set[gr_] = sacc;
            set[64 + gr_] = bnext;
            ptx::named_sync(3, 64);
            if (gr_ >= 32) set[gr_] = sacc + set[31];
            ptx::named_sync(3, 64);
            set[128 + gr_] = fast_exp(set[gr_]);
            set[192 + gr_] = fast_exp(set[63] - set[gr_]);
        };
        // Without warp 8, one thread per tile issues its loads: [K;Q] thread
        // 0, V thread 32, Z thread 64; each loads the next chunk's tile as
        // soon as this chunk is done with it.
        if (!PW && n_chunks > 0) {                   // chunk 0's tiles
            if (tid == 0) issue_qk(0);
            else if (tid == 32) issue_v(0);
            else if (tid == 64) {                    // Z: once the transform grid is done
                asm volatile("griddepcontrol.wait;" ::: "memory");
                issue_z(0);
            }
        }
        if (gate_thread && n_chunks > 0) {
            load_gates(0);
            scan_gates(gsets);
            if (n_chunks > 1) load_gates(1);
        }
        ptx::named_sync(1, NT);

        for (int c = 0; c < n_chunks && !*abort_flag; ++c) {
            const int t0 = c * C;
            const int n = min(C, T - t0);
            const bool more = c + 1 < n_chunks;
            const int sq = c % CF::NQK, sv = c % CF::NVS, sz = c % CF::NZS;
            const uint8_t *sQK = sQK0 + sq * CF::QK_BYTES;
            const uint8_t *sV = sV0 + sv * CF::V_BYTES;
            const uint8_t *sZhi = sZ0 + sz * Z_BYTES, *sZlo = sZhi + 16384;
            const uint32_t aQK = ptx::smem_u32(sQK);
            float *sG = gsets + (c & 1) * 256;        // this chunk's gate set
            float *sBeta = sG + 64;
            float *sGam = sG + 128;
            float *sEnd = sG + 192;

            // ---------------- 1. the chunk's tiles: [K;Q] seen by the threads
            // that read it (thread 0 issues the products, threads 128-191 take
            // the norms), V and Z by thread 64 for everyone, so that thread 0
            // issues the Z R product without a wait of its own.  A wait that
            // gives up sets the abort flag before one of the chunk's barriers,
            // and the loop stops at its next test, all threads together.
            if (tid == 0 || (NORM && tid >= 128 && tid < 192)) {
                if (!ptx::mbar_wait(&bars.full_qk[sq], (uint32_t)((c / CF::NQK) & 1), abort_flag))
                    fail();
            } else if (tid == 64) {
                if (!ptx::mbar_wait(&bars.full_v[sv], (uint32_t)((c / CF::NVS) & 1), abort_flag) ||
                    !ptx::mbar_wait(&bars.full_z[sz], (uint32_t)((c / CF::NZS) & 1), abort_flag))
                    fail();
            }
            ptx::named_sync(1, NT);

            // ---------------- 4. MMA: [K;Q] [S hi | S lo]^T  (M=128, N=2 BV, K=D)
            if (tid == 0) {
                ptx::tc_fence_after();
                constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 2 * BV, false, true);
                const uint32_t bS = ptx::smem_u32(sShi);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t da =
                        ptx::smem_desc(aQK + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    const uint64_t db =
                        ptx::smem_desc(bS + kk * 16 * ROWB, CF::LBO_S, 8 * ROWB, CF::SWZ);
                    ptx::mma_bf16(tmem + CF::COL_X, da, db, idesc, kk > 0);
                }
                ptx::mma_commit(&bars.mma);
            }
            if constexpr (NORM) {                     // 1/|k|, 1/|q| of the chunk's tokens
                if (tid >= 128 && tid < 192) {
                    float kk, qq;
                    qk_row_sumsq<D / 64>(sQK, tid - 128, kk, qq);
                    sNk[tid - 128] = inv_norm(kk);
                    sNq[tid - 128] = inv_norm(qq);
                }
                ptx::named_sync(1, NT);
            }
            wait_mma();

            // ---------------- 5. R = beta V - beta gamma K S^T  (lanes 0-63)
            float xq[HALF];   // Q S^T for this thread's output row (lanes 64-127)
            {
                float x[HALF];
                tmem_ld_pair<HALF>(tmem + lane_off + CF::COL_X + wg * HALF, BV, x);
                if (row < 64) {
                    const int r = row;
                    const float br = sBeta[r], bg = br * (NORM ? sGam[r] * sNk[r] : sGam[r]);
#pragma unroll
                    for (int j = 0; j < HALF; j += 16) {
                        float rr[16];
#pragma unroll
                        for (int e8 = 0; e8 < 16; e8 += 8) {
                            // 8 values of row r: one 16-byte chunk of the swizzled V tile
                            const uint4 raw = *reinterpret_cast<const uint4 *>(
                                sV + ptx::swz_offset<ROWB>(r, wg * HALF + j + e8));
                            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float vv = __uint_as_float(
                                    (e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16));
                                rr[e8 + e] = fmaf(br, vv, -bg * x[j + e8 + e]);
                            }
                        }
                        store_split16<ROWB>(sRhi, sRlo, r, wg * HALF + j, rr);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < HALF; ++j) xq[j] = x[j];
                    if (gate_thread && more) {        // the next chunk's gates
                        scan_gates(gsets + ((c + 1) & 1) * 256);
                        if (c + 2 < n_chunks) load_gates(c + 2);
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_sync(1, NT);
            if (tid == 32) {                          // V of this chunk has been read
                if constexpr (PW) ptx::mbar_arrive(&bars.empty_v[sv]);
                else if (more) issue_v(c + 1);
            }

            // ---------------- 6. MMA: Z R  (M=128, K=64): Z hi [R hi | R lo] (N = 2 BV),
            //                    then Z lo R hi into the hi half
            if (tid == 0) {
                {
                    ptx::tc_fence_after();
                    constexpr uint32_t idesc2 = ptx::idesc_bf16_f32(128, 2 * BV, false, true);
                    constexpr uint32_t idesc1 = ptx::idesc_bf16_f32(128, BV, false, true);
                    const uint32_t aZhi = ptx::smem_u32(sZhi), aZlo = ptx::smem_u32(sZlo);
                    const uint32_t bR = ptx::smem_u32(sRhi);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t db =
                            ptx::smem_desc(bR + kk * 16 * ROWB, CF::LBO_RU, 8 * ROWB, CF::SWZ);
                        ptx::mma_bf16(tmem + CF::COL_Y, ptx::smem_desc(aZhi + kk * 32, 16, 1024),
                                      db, idesc2, kk > 0);
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t db =
                            ptx::smem_desc(bR + kk * 16 * ROWB, CF::LBO_RU, 8 * ROWB, CF::SWZ);
                        ptx::mma_bf16(tmem + CF::COL_Y, ptx::smem_desc(aZlo + kk * 32, 16, 1024),
                                      db, idesc1, true);
                    }
                    ptx::mma_commit(&bars.mma);
                    if constexpr (PW) ptx::mma_commit(&bars.empty_z[sz]);   // Z free once it is done
                }
            }
            wait_mma();
            if (!PW && tid == 64 && more) issue_z(c + 1); // the Z R product has read Z

            // ---------------- 7. O (lanes 64-127) and U~ hi / lo (lanes 0-63)
            {
                float y[HALF];
                tmem_ld_pair<HALF>(tmem + lane_off + CF::COL_Y + wg * HALF, BV, y);
                if (row >= 64) {
                    const int r = row - 64;
                    if (r < n) {
                        const float gr = NORM ? sGam[r] * sNq[r] : sGam[r];
                        // output element of (token t0 + r, value v0 + wg * HALF)
                        const size_t oi = ((size_t)b * T + t0 + r) * tok_stride + (size_t)h * D +
                                          v0 + wg * HALF;
#pragma unroll
                        for (int j = 0; j < HALF; j += 4) {
                            float4 o4;
                            o4.x = fmaf(gr, xq[j + 0], y[j + 0]) * scale;
                            o4.y = fmaf(gr, xq[j + 1], y[j + 1]) * scale;
                            o4.z = fmaf(gr, xq[j + 2], y[j + 2]) * scale;
                            o4.w = fmaf(gr, xq[j + 3], y[j + 3]) * scale;
                            if (out_bf16) {                // 4 values rounded to nearest even
                                const __nv_bfloat162 lo = __floats2bfloat162_rn(o4.x, o4.y);
                                const __nv_bfloat162 hi = __floats2bfloat162_rn(o4.z, o4.w);
                                uint2 w;
                                w.x = *reinterpret_cast<const uint32_t *>(&lo);
                                w.y = *reinterpret_cast<const uint32_t *>(&hi);
                                *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(out) +
                                                           oi + j) = w;
                            } else {
                                *reinterpret_cast<float4 *>(out + oi + j) = o4;
                            }
                        }
                    }
                } else {
                    const int r = row;
                    const float er = NORM ? sEnd[r] * sNk[r] : sEnd[r];
#pragma unroll
                    for (int j = 0; j < HALF; j += 16) {
                        float u[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) u[e] = er * y[j + e];
                        store_split16<ROWB>(sRhi, sRlo, r, wg * HALF + j, u);   // R no longer needed
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_sync(1, NT);

            // ---------------- 8. MMA: K^T [U~ hi | U~ lo]  (per 128-key tile: M=128,
            //                    N=2 BV, K=64)
            if (tid == 0) {
                ptx::tc_fence_after();
                constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 2 * BV, true, true);
                const uint32_t bU = ptx::smem_u32(sRhi);
#pragma unroll
                for (int kt = 0; kt < KT; ++kt) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t da =
                            ptx::smem_desc(aQK + kt * 2 * 16384 + kk * 2048, 16384, 1024);
                        const uint64_t db =
                            ptx::smem_desc(bU + kk * 16 * ROWB, CF::LBO_RU, 8 * ROWB, CF::SWZ);
                        ptx::mma_bf16(tmem + CF::COL_DS + kt * 2 * BV, da, db, idesc, kk > 0);
                    }
                }
                ptx::mma_commit(&bars.mma);
                if constexpr (PW) ptx::mma_commit(&bars.empty_qk[sq]);   // both products read [K;Q]
            }
            wait_mma();
            if (!PW && tid == 0 && more) issue_qk(c + 1); // both products have read [K;Q]

            // ---------------- 9. S = gamma_C S + dS^T; S hi / lo for the next chunk
            {
                const float gC = sGam[63];
#pragma unroll
                for (int kt = 0; kt < KT; ++kt) {
                    float ds[HALF];
                    tmem_ld_pair<HALF>(tmem + lane_off + CF::COL_DS + kt * 2 * BV + wg * HALF, BV,
                                       ds);
                    const int key = kt * 128 + row;
#pragma unroll
                    for (int j = 0; j < HALF; ++j) S[kt][j] = fmaf(gC, S[kt][j], ds[j]);
                    if (key < D) {
#pragma unroll
                        for (int j = 0; j < HALF; j += 16) {
                            float x[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) x[e] = S[kt][j + e];
                            store_split16<ROWB>(sShi, sSlo, key, wg * HALF + j, x);
                        }
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_sync(1, NT);
            ptx::tc_fence_after();
        }

        if (!PW && (tid == 0 || tid == 32 || tid == 64)) drain();

        // ---- final state block
        if (!*abort_flag) {
#pragma unroll
            for (int kt = 0; kt < KT; ++kt) {
                const int key = kt * 128 + row;
                if (key < D) {
#pragma unroll
                    for (int j = 0; j < HALF; ++j) {
                        const int v = v0 + wg * HALF + j;
                        state_out[st_base + (size_t)v * D + key] = S[kt][j];
                    }
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, CF::TMEM_COLS);
}
// ---------------------------------------------------------------------------
// head_dim 64 and 128: one CTA per (sequence, head) owns every value row, so
// the chunk-local UT transform is built once per chunk and head.  The state
// is held transposed with respect to chunked_kernel: TMEM lanes are value
// rows and columns are keys, so it accumulates in place (S += U~^T K) and its
// bf16 hi / lo split feeds the next chunk's MMA straight from TMEM (A
// operand).  Two warp-specialised streams share the CTA:
//   transform stream (warps 8-15), chunk c, one chunk ahead of the other:
//     [K;Q] K^T (M = 128) -> A (fp32), P (hi / lo) -> T = (I + A)^-1 in
//     place -> T (hi / lo) into Z rows 0-63 -> P T (A = [P hi; P lo],
//     B = T, MN-major) -> P T (hi / lo) into Z rows 64-127
//   state stream (warps 0-7), chunk c (M = 128 value rows in every product):
//     X^T  = S [K;Q]^T             (A = S hi / lo in TMEM, B = [K;Q] from TMA)
//     R^T  = beta V^T - beta gamma (K S^T)^T                   (CUDA cores)
//     [U^T | (P U)^T] = R^T Z^T    (one N = 128 product, B = Z rows)
//     S   += (diag(exp(G_C - G)) U)^T K   (S pre-scaled by gamma_C; B = K MN-major)
//     O    = (gamma Q S^T + P U) / sqrt(d): staged in shared memory (at
//            head_dim 128 in the chunk's Z buffer, while the S product
//            runs), one TMA store per chunk
// The streams hand over through mbarriers: TMA stage full, V full, gates
// ready (4 sets), Z ready / Z free (2 buffers), and each stream's MMA
// completions.  For head_dim 64 the same code runs with TMEM lanes 64-127
// carrying no value row (their results are never read).
namespace d128 {

constexpr int NS = 256;                 // threads per stream
constexpr int NTH = 2 * NS;             // state stream (warps 0-7) + transform stream (8-15)
constexpr int BAR_S = 1, BAR_Z = 2;     // hardware barrier of each stream
// Thread of the transform stream that issues its products and mbarrier
// arrivals: warp 10, SMSP 2.  The state stream's issuing thread (0) sits on
// SMSP 0, and a warp blocked issuing holds back the other warps of its SMSP
// (measured, 8 x 16384 x 64 x 64: 5.05 -> 4.98 ms against thread 0 of the
// stream, no change on SMSP 1).
constexpr int ZI = 64;
// shared memory map (bytes from a 1024-aligned base)
constexpr int OFF_QK = 0;               // 2 stages x [K;Q] (2 slabs x 128 rows x 128 B)
constexpr int OFF_V = 65536;            // V of one chunk (2 boxes x 64 rows x 128 B)
constexpr int OFF_Z = 81920;            // 2 buffers x {Z hi, Z lo} (128 rows x 128 B each)
constexpr int OFF_PP = 147456;          // P hi (rows 0-63) | P lo (rows 64-127)
constexpr int OFF_AT = 163840;          // A, then T in place: fp32 64 x FST
constexpr int OFF_W = OFF_AT + 64 * FST * 4;   // 16 x 96 or 32 x 40 fp32
constexpr int OFF_RT = 187392;          // R^T (then U~^T) hi | lo: 128 rows x 128 B each
constexpr int OFF_G = OFF_RT + 32768;   // 4 gate sets of GS floats (layout at scan_gates)
constexpr int GS = 512;                 // floats per gate set
constexpr int SMEM = OFF_G + 4 * GS * 4 + 1024;
static_assert(OFF_W + 16 * 96 * 4 <= OFF_RT && 16 * 96 >= 32 * 40, "scratch overlaps R^T");
static_assert(OFF_PP + 24576 <= OFF_RT, "P lo rows 64-127 are read from the scratch");
static_assert(SMEM + 256 <= 232448, "shared memory (dynamic + static)");
// TMEM columns
constexpr uint32_t C_SACC = 0;    // S (fp32): lane = value, column = key
constexpr uint32_t C_SHI = 128;   // S hi, bf16 pairs (keys 2c, 2c+1 in column c)
constexpr uint32_t C_SLO = 192;   // S lo
constexpr uint32_t C_Y = 256;     // [U^T | (P U)^T] (128 columns, one MMA); PU half = K part of X
constexpr uint32_t C_U = 256;     //   U^T
constexpr uint32_t C_PU = 320;    //   (P U)^T
constexpr uint32_t C_X = 320;     // X^T: columns 0-63 K part (consumed before C_PU is written),
                                  //      64-127 Q part (columns 384-447)
constexpr uint32_t C_KQ = 448;    // [K;Q] K^T, then P T (lanes 0-63): transform stream only

struct Shared {
    uint64_t qk_full[2];   // TMA: [K;Q] of the chunk in the stage has landed
    uint64_t v_full;       // TMA: V of the chunk has landed
    uint64_t z_ready[2];   // transform stream: Z = [T; P T] of the chunk is in its buffer
    uint64_t z_free[2];    // state stream: the Z R product (and, at head_dim 128, the O
                           // store that reuses the buffer) have finished reading it
    uint64_t g_ready[4];   // transform stream: the chunk's gate set is written
    uint64_t mma_s, mma_z; // each stream's MMA completions
    uint32_t tmem_base;
    int abort;
};

constexpr float LOG2E = 1.4426950408889634f;

// 2^x; results below the fp32 normal range flush to zero (a decay factor
// under 1e-38 is zero for every purpose here).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Gates of one chunk, held by threads 0-63 between the global loads and
// the scan: lane l of warp w keeps g of tokens l and 32 + l (0 past T) and
// beta of its own token w*32 + l.
struct GateRegs {
    float ga, gb, bown;
};

__device__ __forceinline__ void load_gates(GateRegs &r, const float *g, const float *beta, int b,
                                           int h, int T, int H, int c, int t) {
    const int t0 = c * C;
    const int n = min(C, T - t0);
    const int l = t & 31;
    const size_t base = ((size_t)b * T + t0) * H + h;
    r.ga = (l < n) ? g[base + (size_t)l * H] : 0.f;
    r.gb = (32 + l < n) ? g[base + (size_t)(32 + l) * H] : 0.f;
    r.bown = (t < n) ? beta[base + (size_t)t * H] : 0.f;
}

// Gate set of one chunk, 8 x 64 floats indexed by token:
//   [0]   G2    = G log2 e, G the inclusive cumsum of max(g, -30)
//   [64]  beta
//   [128] gamma = exp(G)
//   [192] end   = exp(G_63 - G) nk       (scales U for the state update)
//   [256] gk    = gamma nk               (the K S^T term of R)
//   [320] gq    = gamma nq               (the Q S^T term of O)
//   [384] nk, [448] nq: 1 / |k|, 1 / |q| with q / k normalisation, else 1.
// scan_gates writes [0, 192) and returns the token's end decay; set_norms
// writes the rest once the chunk's [K;Q] tiles have landed.  Threads 0-63 of
// a stream (t), no barrier inside.
__device__ __forceinline__ float scan_gates(const GateRegs &r, float *gs, int t) {
    const int l = t & 31;
    float sa = fmaxf(r.ga, -30.f), sb = fmaxf(r.gb, -30.f);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float ya = __shfl_up_sync(0xffffffffu, sa, o);
        const float yb = __shfl_up_sync(0xffffffffu, sb, o);
        if (l >= o) { sa += ya; sb += yb; }
    }
    const float tot0 = __shfl_sync(0xffffffffu, sa, 31);
    const float tot = tot0 + __shfl_sync(0xffffffffu, sb, 31);
    const float G = (t < 32) ? sa : tot0 + sb;
    gs[t] = G * LOG2E;
    gs[64 + t] = r.bown;
    gs[128 + t] = ex2(G * LOG2E);
    return ex2((tot - G) * LOG2E);
}

template <int NSLAB, bool NORM>
__device__ __forceinline__ void set_norms(float *gs, const uint8_t *qk, int t, float end) {
    float nk = 1.f, nq = 1.f;
    if constexpr (NORM) {
        float kk, qq;
        qk_row_sumsq<NSLAB>(qk, t, kk, qq);
        nk = inv_norm(kk);
        nq = inv_norm(qq);
    }
    const float gam = gs[128 + t];
    gs[192 + t] = end * nk;
    gs[256 + t] = gam * nk;
    gs[320 + t] = gam * nq;
    gs[384 + t] = nk;
    gs[448 + t] = nq;
}

// 32 consecutive keys of one state row: hi / lo pairs -> 16 + 16 packed TMEM
// columns, gamma * S -> 32 fp32 columns.
__device__ __forceinline__ void put_state32(uint32_t tmem_lane, int key0, float (&x)[32],
                                            float gamma) {
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) ptx::split_pair(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
    ptx::tmem_st16(tmem_lane + C_SHI + key0 / 2, hi);
    ptx::tmem_st16(tmem_lane + C_SLO + key0 / 2, lo);
#pragma unroll
    for (int e = 0; e < 16; ++e) hi[e] = __float_as_uint(gamma * x[e]);
    ptx::tmem_st16(tmem_lane + C_SACC + key0, hi);
#pragma unroll
    for (int e = 0; e < 16; ++e) lo[e] = __float_as_uint(gamma * x[16 + e]);
    ptx::tmem_st16(tmem_lane + C_SACC + key0 + 16, lo);
}

template <int D, bool NORM>
__global__ void __launch_bounds__(NTH, 1)
chunked_d128_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, const float *__restrict__ g,
                    const float *__restrict__ beta, const float *state_in, float *state_out,
                    float *__restrict__ out, int T, int H, int Hk, float scale,
                    int *status, bool out_bf16)
{
    // Where O is staged.  head_dim 128: in the chunk's Z buffer, so that it
    // overlaps the S product, which still reads the R^T / U~^T buffer; the
    // buffer then returns to the transform stream only after the O store has
    // read it.  head_dim 64, where the transform stream limits the chunk: in
    // the R^T buffer after the S product, so that Z buffers return as soon as
    // the Z R product has read them.  (Measured: each choice is the faster
    // one at its head_dim.)
    constexpr bool kOInZ = (D == 128);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ Shared sh;
    float *sAT = reinterpret_cast<float *>(sm + OFF_AT);
    float *sW = reinterpret_cast<float *>(sm + OFF_W);
    float *gsets = reinterpret_cast<float *>(sm + OFF_G);
    uint8_t *sPhi = sm + OFF_PP, *sPlo = sm + OFF_PP + 8192;
    uint8_t *sRhi = sm + OFF_RT, *sRlo = sm + OFF_RT + 16384;
    uint8_t *sV = sm + OFF_V;

    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    constexpr int NSLAB = D / 64;            // 64-key slabs of [K;Q] and 64-value boxes of V
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const bool zstream = tid >= NS;          // transform stream
    const int t = tid & (NS - 1);            // thread index within the stream
    const int wg = t >> 7;                   // which half of the columns this thread handles
    const int row = t & 127;                 // TMEM lane: value row, or [K;Q] row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int bh = blockIdx.x;
    const int b = bh / H, h = bh - b * H;
    const int n_chunks = (T + C - 1) / C;
    const size_t st_base = (size_t)bh * D * D;

    if (tid == 0) {
        sh.abort = 0;
        ptx::mbar_init(&sh.qk_full[0], 1);
        ptx::mbar_init(&sh.qk_full[1], 1);
        ptx::mbar_init(&sh.v_full, 1);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sh.z_ready[i], 1);
            ptx::mbar_init(&sh.z_free[i], 1);
        }
        for (int i = 0; i < 4; ++i) ptx::mbar_init(&sh.g_ready[i], 1);
        ptx::mbar_init(&sh.mma_s, 1);
        ptx::mbar_init(&sh.mma_z, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
        ptx::prefetch_tmap(&tm_o);
    }
    if (warp == 0) {
        ptx::tmem_alloc(&sh.tmem_base, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const uint32_t tl = tmem + lane_off;     // this warp's lane quarter
    volatile int *abort_flag = &sh.abort;
    uint32_t mma_phase = 0;

    auto fail = [&]() {
        if (atomicExch(const_cast<int *>(abort_flag), 1) == 0) atomicExch(status, GDN_ERR_TIMEOUT);
    };
    auto wait = [&](uint64_t *bar, uint32_t parity) {
        if (!ptx::mbar_wait(bar, parity, abort_flag)) fail();
    };
    auto issue_qk = [&](int c) {
        const int st = c & 1;
        uint8_t *qk = sm + OFF_QK + st * 32768;
        ptx::mbar_arrive_expect_tx(&sh.qk_full[st], NSLAB * 2 * 8192);
#pragma unroll
        for (int s = 0; s < NSLAB; ++s) {
            ptx::tma_load_4d(qk + s * 16384, &tm_k, &sh.qk_full[st], s * 64, h % Hk, c * C, b);
            ptx::tma_load_4d(qk + s * 16384 + 8192, &tm_q, &sh.qk_full[st], s * 64, h % Hk, c * C,
                             b);
        }
    };
    auto issue_v = [&](int c) {
        ptx::mbar_arrive_expect_tx(&sh.v_full, NSLAB * 8192);
#pragma unroll
        for (int s = 0; s < NSLAB; ++s)
            ptx::tma_load_4d(sV + s * 8192, &tm_v, &sh.v_full, s * 64, h, c * C, b);
    };
    // The same loads split over one thread in each of warps 0-3 (the state
    // stream issues them mid-chunk, where a single thread would hold up the
    // products it also issues): box i of [K;Q] (K slab 0, Q slab 0, K slab
    // 1, Q slab 1) and of V by thread 32 i.  Thread 0 arms the barrier for
    // the whole tile; a box that lands before that leaves the transaction
    // count negative, which keeps the phase open until the rest has landed.
    auto issue_qk_part = [&](int c, int i) {
        const int st = c & 1;
        uint8_t *qk = sm + OFF_QK + st * 32768;
        if (i == 0) ptx::mbar_arrive_expect_tx(&sh.qk_full[st], NSLAB * 2 * 8192);
        if (i < 2 * NSLAB)
            ptx::tma_load_4d(qk + (i >> 1) * 16384 + (i & 1) * 8192, (i & 1) ? &tm_q : &tm_k,
                             &sh.qk_full[st], (i >> 1) * 64, h % Hk, c * C, b);
    };
    auto issue_v_part = [&](int c, int i) {
        if (i == 0) ptx::mbar_arrive_expect_tx(&sh.v_full, NSLAB * 8192);
        if (i < NSLAB) ptx::tma_load_4d(sV + i * 8192, &tm_v, &sh.v_full, i * 64, h, c * C, b);
    };
    if (tid == 0) {
        issue_qk(0);
        if (n_chunks > 1) issue_qk(1);
        issue_v(0);
    }

    if (zstream) {
        // ================= transform stream: Z = [T; P T] of every chunk
        GateRegs gr{0.f, 0.f, 0.f};          // gates of the chunk about to start
        if (t < 64) load_gates(gr, g, beta, b, h, T, H, 0, t);
        for (int c = 0; c < n_chunks; ++c) {
            const int st = c & 1;
            const uint32_t aQK = ptx::smem_u32(sm + OFF_QK + st * 32768);
            float *gs = gsets + (c & 3) * GS;
            const float *sG = gs, *sBeta = gs + 64, *sNk = gs + 384, *sNq = gs + 448;
            uint8_t *sZhi = sm + OFF_Z + st * 32768, *sZlo = sZhi + 16384;

            float end = 0.f;
            if (t < 64) {
                end = scan_gates(gr, gs, t);
                if (c + 1 < n_chunks) load_gates(gr, g, beta, b, h, T, H, c + 1, t);
            }
            wait(&sh.qk_full[st], (uint32_t)((c >> 1) & 1));
            if (t < 64) set_norms<NSLAB, NORM>(gs, sm + OFF_QK + st * 32768, t, end);
            ptx::named_sync(BAR_Z, NS);
            const bool ok = !*abort_flag;
            if (t == ZI) {
                ptx::mbar_arrive(&sh.g_ready[c & 3]);
                // [K;Q] K^T  (M = 128, N = 64, K = 128)
                if (ok) {
                    ptx::tc_fence_after();
                    constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 64, false, false);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t da =
                            ptx::smem_desc(aQK + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                        ptx::mma_bf16(tmem + C_KQ, da, da, idesc, kk > 0);
                    }
                    ptx::mma_commit(&sh.mma_z);
                }
            }
            wait(&sh.mma_z, mma_phase);
            mma_phase ^= 1;
            ptx::tc_fence_after();

            // A (rows 0-63) as fp32; P (rows 64-127) as hi / lo rows; with q / k
            // normalisation A[r,i] and P[r,i] carry nk_r nk_i and nq_r nk_i
            {
                const int r = row & 63;
                const float Gr = sG[r];
                const float br = NORM ? sBeta[r] * sNk[r] : sBeta[r];
                const float pr = NORM ? sNq[r] : 1.f;
#pragma unroll 1
                for (int jc = wg * 32; jc < wg * 32 + 32; jc += 16) {
                    float kq[16];
                    ptx::tmem_ld16(tl + C_KQ + jc, kq);
                    ptx::tmem_ld_wait();
                    const float4 *g4 = reinterpret_cast<const float4 *>(sG + jc);
                    float gi[16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 v4 = g4[q];
                        gi[4 * q] = v4.x; gi[4 * q + 1] = v4.y; gi[4 * q + 2] = v4.z; gi[4 * q + 3] = v4.w;
                    }
                    if constexpr (NORM) {             // column factor nk_i into the K K^T / Q K^T entries
                        const float4 *n4 = reinterpret_cast<const float4 *>(sNk + jc);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 v4 = n4[q];
                            kq[4 * q] *= v4.x; kq[4 * q + 1] *= v4.y;
                            kq[4 * q + 2] *= v4.z; kq[4 * q + 3] *= v4.w;
                        }
                    }
                    if (row < 64) {
                        float a[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int i = jc + j;
                            a[j] = (i < r) ? br * ex2(Gr - gi[j]) * kq[j] : 0.f;
                        }
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4 *>(sAT + r * FST + jc + j) =
                                make_float4(a[j], a[j + 1], a[j + 2], a[j + 3]);
                    } else {
                        float p[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int i = jc + j;
                            p[j] = (i <= r) ? pr * ex2(Gr - gi[j]) * kq[j] : 0.f;
                        }
                        ptx::store_split8(sPhi, sPlo, r, jc, p);
                        ptx::store_split8(sPhi, sPlo, r, jc + 8, p + 8);
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_sync(BAR_Z, NS);

            // T = (I + A)^-1 in place
            if constexpr (D == 128) ut_transform32(sAT, sW, t, BAR_Z);
            else ut_transform16(sAT, sW, t, BAR_Z);

            // T as hi / lo into rows 0-63 of this chunk's Z buffer, once the
            // state stream has finished with the chunk that used it before
            if (c >= 2) wait(&sh.z_free[st], (uint32_t)(((c - 2) >> 1) & 1));
            {
                const int r = t >> 2, c0 = (t & 3) * 16;
                float tv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) tv[e] = sAT[r * FST + c0 + e];
                ptx::store_split8(sZhi, sZlo, r, c0, tv);
                ptx::store_split8(sZhi, sZlo, r, c0 + 8, tv + 8);
            }
            ptx::fence_proxy_async_smem();
            ptx::named_sync(BAR_Z, NS);

            // P T  (A = [P hi; P lo] 128 rows, B = T rows (MN-major), N = 64, K = 64)
            if (t == ZI && !*abort_flag) {
                ptx::tc_fence_after();
                constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 64, false, true);
                const uint32_t aP[3] = {ptx::smem_u32(sPhi), ptx::smem_u32(sPhi), ptx::smem_u32(sPlo)};
                const uint32_t bT[3] = {ptx::smem_u32(sZhi), ptx::smem_u32(sZlo), ptx::smem_u32(sZhi)};
#pragma unroll
                for (int part = 0; part < 3; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_bf16(tmem + C_KQ, ptx::smem_desc(aP[part] + kk * 32, 16, 1024),
                                      ptx::smem_desc(bT[part] + kk * 2048, 8192, 1024), idesc,
                                      part > 0 || kk > 0);
                ptx::mma_commit(&sh.mma_z);
            }
            wait(&sh.mma_z, mma_phase);
            mma_phase ^= 1;
            ptx::tc_fence_after();

            // P T rows -> Z rows 64-127 (TMEM lanes 0-63)
            if ((warp & 3) < 2) {
#pragma unroll 1
                for (int jc = wg * 32; jc < wg * 32 + 32; jc += 16) {
                    float pt[16];
                    ptx::tmem_ld16(tl + C_KQ + jc, pt);
                    ptx::tmem_ld_wait();
                    ptx::store_split8(sZhi, sZlo, 64 + row, jc, pt);
                    ptx::store_split8(sZhi, sZlo, 64 + row, jc + 8, pt + 8);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_sync(BAR_Z, NS);
            if (t == ZI) ptx::mbar_arrive(&sh.z_ready[st]);
        }
    } else {
        // ================= state stream
        // initial state: thread (value row, key half) -> TMEM, pre-scaled by
        // the first chunk's gamma_C for the in-place accumulation
        wait(&sh.g_ready[0], 0);
        const bool vrow = row < D;               // this lane is a value row of the state
        if (vrow) {
            const float gC = gsets[128 + 63];
#pragma unroll 1
            for (int kg = 0; kg < D / 2; kg += 32) {
                const int key0 = wg * (D / 2) + kg;
                float x[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (state_in)
                        t4 = *reinterpret_cast<const float4 *>(state_in + st_base +
                                                               (size_t)row * D + key0 + e);
                    x[e] = t4.x; x[e + 1] = t4.y; x[e + 2] = t4.z; x[e + 3] = t4.w;
                }
                put_state32(tl, key0, x, gC);
            }
            ptx::tmem_st_wait();
        }
        ptx::tc_fence_before();
        ptx::named_sync(BAR_S, NS);

        // O of a chunk into `stage` (32 KB or 16 KB, 1024-aligned) and out by
        // one TMA store; TMEM columns read: X^T's Q half and (P U)^T
        auto o_epilogue = [&](uint8_t *stage, const float *sGam, int t0) {
            if constexpr (kOInZ) ptx::tc_fence_after();   // else done after the S wait
            if (vrow) {
                const int v = row;
                float *ot = reinterpret_cast<float *>(stage);
                __nv_bfloat16 *otb = reinterpret_cast<__nv_bfloat16 *>(stage);
#pragma unroll 1
                for (int jc = wg * 32; jc < wg * 32 + 32; jc += 16) {
                    float xq[16], pu[16], gm[16];
                    ptx::tmem_ld16(tl + C_X + 64 + jc, xq);
                    ptx::tmem_ld16(tl + C_PU + jc, pu);
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float4 g4 = *reinterpret_cast<const float4 *>(sGam + jc + j);
                        gm[j] = g4.x; gm[j + 1] = g4.y; gm[j + 2] = g4.z; gm[j + 3] = g4.w;
                    }
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float o = fmaf(gm[j], xq[j], pu[j]) * scale;
                        if (out_bf16) otb[(jc + j) * D + v] = __float2bfloat16_rn(o);
                        else ot[(jc + j) * D + v] = o;
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::named_sync(BAR_S, NS);
            if (t == 64) {                             // thread 64 owns the O stores
                ptx::tma_store_4d(&tm_o, stage, 0, h, t0, b);
                ptx::bulk_commit_group();
            }
        };

        for (int c = 0; c < n_chunks; ++c) {
            const int st = c & 1;
            const int t0 = c * C;
            const int n = min(C, T - t0);
            const bool last = (c + 1 == n_chunks);
            const float *gs = gsets + (c & 3) * GS;
            // gamma nk for R, gamma nq for O, end nk for U~ (nk = nq = 1 unless
            // q and k are normalised)
            const float *sBeta = gs + 64, *sGamK = gs + 256, *sGamQ = gs + 320, *sEnd = gs + 192;
            const uint32_t aQK = ptx::smem_u32(sm + OFF_QK + st * 32768);
            uint8_t *sZhi = sm + OFF_Z + st * 32768, *sZlo = sZhi + 16384;

            wait(&sh.g_ready[c & 3], (uint32_t)((c >> 2) & 1));
            wait(&sh.qk_full[st], (uint32_t)((c >> 1) & 1));

            // X^T = S [K;Q]^T  (A = S hi / lo from TMEM, M = 128, N = 128, K = 128)
            if (t == 0) {
                ptx::tc_fence_after();
                constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 128, false, false);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        ptx::mma_bf16_ts(tmem + C_X, tmem + (part ? C_SLO : C_SHI) + kk * 8,
                                         ptx::smem_desc(aQK + (kk >> 2) * 16384 + (kk & 3) * 32,
                                                        16, 1024),
                                         idesc, part > 0 || kk > 0);
                ptx::mma_commit(&sh.mma_s);
            }
            wait(&sh.mma_s, mma_phase);
            mma_phase ^= 1;
            ptx::tc_fence_after();

            // R^T = beta V^T - beta gamma (K S^T)^T  (value row v, tokens of this half)
            wait(&sh.v_full, (uint32_t)(c & 1));
            if (vrow) {
                const int v = row;
                const uint8_t *vbox = sV + (v >> 6) * 8192;
#pragma unroll 1
                for (int jc = wg * 32; jc < wg * 32 + 32; jc += 16) {
                    float x[16];
                    ptx::tmem_ld16(tl + C_X + jc, x);
                    ptx::tmem_ld_wait();
                    float rr[16], bt[16], gm[16];
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float4 b4 = *reinterpret_cast<const float4 *>(sBeta + jc + j);
                        const float4 g4 = *reinterpret_cast<const float4 *>(sGamK + jc + j);
                        bt[j] = b4.x; bt[j + 1] = b4.y; bt[j + 2] = b4.z; bt[j + 3] = b4.w;
                        gm[j] = g4.x; gm[j + 1] = g4.y; gm[j + 2] = g4.z; gm[j + 3] = g4.w;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tk = jc + j;
                        const float vv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                            vbox + ptx::sw128_offset(tk, v & 63)));
                        rr[j] = bt[j] * (vv - gm[j] * x[j]);
                    }
                    ptx::store_split8(sRhi, sRlo, v, jc, rr);
                    ptx::store_split8(sRhi, sRlo, v, jc + 8, rr + 8);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_sync(BAR_S, NS);
            if (!last && (t & 31) == 0 && t < 32 * NSLAB) issue_v_part(c + 1, t >> 5);   // V consumed

            // [U^T | (P U)^T] = R^T Z^T with Z = [T; P T]: one N = 128 product
            wait(&sh.z_ready[st], (uint32_t)((c >> 1) & 1));
            if (t == 0) {
                ptx::tc_fence_after();
                constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, 128, false, false);
                const uint32_t aR[3] = {ptx::smem_u32(sRhi), ptx::smem_u32(sRhi), ptx::smem_u32(sRlo)};
                const uint32_t bZ[3] = {ptx::smem_u32(sZhi), ptx::smem_u32(sZlo), ptx::smem_u32(sZhi)};
#pragma unroll
                for (int part = 0; part < 3; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_bf16(tmem + C_Y, ptx::smem_desc(aR[part] + kk * 32, 16, 1024),
                                      ptx::smem_desc(bZ[part] + kk * 32, 16, 1024), idesc,
                                      part > 0 || kk > 0);
                ptx::mma_commit(&sh.mma_s);
                if constexpr (!kOInZ) ptx::mma_commit(&sh.z_free[st]);
            }
            wait(&sh.mma_s, mma_phase);
            mma_phase ^= 1;
            ptx::tc_fence_after();

            // U~^T hi / lo first: it is all the state update needs
            if (vrow) {
                const int v = row;
#pragma unroll 1
                for (int jc = wg * 32; jc < wg * 32 + 32; jc += 16) {
                    float u[16], en[16];
                    ptx::tmem_ld16(tl + C_U + jc, u);
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float4 e4 = *reinterpret_cast<const float4 *>(sEnd + jc + j);
                        en[j] = e4.x; en[j + 1] = e4.y; en[j + 2] = e4.z; en[j + 3] = e4.w;
                    }
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) u[j] *= en[j];
                    ptx::store_split8(sRhi, sRlo, v, jc, u);
                    ptx::store_split8(sRhi, sRlo, v, jc + 8, u + 8);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::named_sync(BAR_S, NS);

            // S += U~^T K  (M = 128 values, N = D keys, K = 64 tokens)
            if (t == 0) {
                ptx::tc_fence_after();
                constexpr uint32_t idesc = ptx::idesc_bf16_f32(128, D, false, true);
                const uint32_t aU[2] = {ptx::smem_u32(sRhi), ptx::smem_u32(sRlo)};
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_bf16(tmem + C_SACC, ptx::smem_desc(aU[part] + kk * 32, 16, 1024),
                                      ptx::smem_desc(aQK + kk * 2048, 16384, 1024), idesc, true);
                ptx::mma_commit(&sh.mma_s);
            }

            // O = (gamma Q S^T + P U) / sqrt(d), staged as a [token][value]
            // fp32 tile and written by one TMA store that clips tokens past T
            if constexpr (kOInZ) {
                o_epilogue(sZhi, sGamQ, t0);  // while the S product runs (it writes only S)
                wait(&sh.mma_s, mma_phase);
                mma_phase ^= 1;
                ptx::tc_fence_after();
            } else {
                wait(&sh.mma_s, mma_phase);
                mma_phase ^= 1;
                ptx::tc_fence_after();
                o_epilogue(sRhi, sGamQ, t0);  // the S product has finished reading U~
            }
            // this stage is free: bring chunk c + 2 into it
            if (c + 2 < n_chunks && (t & 31) == 0 && t < 64 * NSLAB) issue_qk_part(c + 2, t >> 5);

            // S: split for the next chunk's X^T and pre-scale by its gamma_C,
            // or write the final state
            float gC = 1.f;
            if (!last) {
                wait(&sh.g_ready[(c + 1) & 3], (uint32_t)(((c + 1) >> 2) & 1));
                gC = gsets[((c + 1) & 3) * GS + 128 + 63];
            }
#pragma unroll 1
            for (int kg = 0; kg < (vrow ? D / 2 : 0); kg += 32) {
                const int key0 = wg * (D / 2) + kg;
                float x[32];
                ptx::tmem_ld16(tl + C_SACC + key0, *reinterpret_cast<float(*)[16]>(x));
                ptx::tmem_ld16(tl + C_SACC + key0 + 16, *reinterpret_cast<float(*)[16]>(x + 16));
                ptx::tmem_ld_wait();
                if (last) {
                    float *dst = state_out + st_base + (size_t)row * D + key0;
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(dst + e) =
                            make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
                } else {
                    put_state32(tl, key0, x, gC);
                }
            }
            if (!last && vrow) ptx::tmem_st_wait();
            if (t == 64) {
                ptx::bulk_wait_read_all();               // the O tile has left its buffer
                if constexpr (kOInZ) ptx::mbar_arrive(&sh.z_free[st]);
            }
            ptx::tc_fence_before();
            ptx::named_sync(BAR_S, NS);
        }
        if (t == 64) ptx::bulk_wait_all();
        // every load addressed to this CTA's shared memory has landed before
        // it exits (on the normal path these phases completed long ago; after
        // a wait gave up they may not have)
        if (t == 0) {
            const volatile int never = 0;
            for (int c = (n_chunks > 2 ? n_chunks - 2 : 0); c < n_chunks; ++c)
                ptx::mbar_wait(&sh.qk_full[c & 1], (uint32_t)((c >> 1) & 1), &never, 1000000000LL);
            if (n_chunks > 0)
                ptx::mbar_wait(&sh.v_full, (uint32_t)((n_chunks - 1) & 1), &never, 1000000000LL);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) ptx::tmem_dealloc(tmem, 512);
}

}  // namespace d128

// ------------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 4-D map over a (B, T, H, d) bf16 tensor; box = {box0 elements of d, 1 head,
// 64 tokens, 1 sequence}, box0 * 2 bytes = the swizzle span (128 B: box0 64,
// 64 B: box0 32).  Tokens past T read as zeros.
bool make_map(CUtensorMap *map, const void *base, int B, int T, int H, int d, int box0) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                   (cuuint64_t)T * H * d * 2};
    const cuuint32_t box[4] = {(cuuint32_t)box0, 1, (cuuint32_t)C, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               box0 == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// 4-D map over the (B, T, H, d) output, fp32 or bf16; box = {d, 1 head, 64
// tokens, 1 sequence}, unswizzled: a [token][value] tile of one chunk.
// Tokens past T are clipped by the store.
bool make_map_out(CUtensorMap *map, void *base, int B, int T, int H, int d, bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t es = bf16 ? 2 : 4;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * es, (cuuint64_t)H * d * es,
                                   (cuuint64_t)T * H * d * es};
    const cuuint32_t box[4] = {(cuuint32_t)d, 1, (cuuint32_t)C, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
               base, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

// Value blocks of the two-kernel state walk for P (sequence, head) pairs on
// `sms` SMs (one walk CTA per SM):
//   - 32 rows for every pair where D / 32 CTAs per pair fit one wave: a small
//     problem then runs twice the CTAs, each with a shorter chain per chunk;
//   - otherwise 64 rows; when that leaves a partial last wave whose pairs fit
//     one wave at 32 rows, the pairs of the full waves keep 64-row blocks and
//     the rest run after them at 32 rows (a shorter last wave: at 8 x 16384
//     tokens x 16 heads x 256, 3 full waves of 64-row blocks and 112 CTAs of
//     32-row blocks instead of a fourth wave of 56 CTAs).
// The walk's kernel launches are then one (pairs64 == 0 or == P) or two.
WalkSplit walk_split(long long P, int D, int sms) {
    WalkSplit w{0};
    if (P <= 0 || sms <= 0) return w;
    const long long per32 = D / 32, per64 = D / 64;
    if (P * per32 <= sms) return w;                          // all 32-row blocks
    w.pairs64 = (int)P;
    const long long ctas64 = P * per64;
    const long long full = ctas64 / sms;
    if (full >= 1 && ctas64 % sms != 0 && (full * sms) % per64 == 0) {
        const long long p64 = full * sms / per64;
        if ((P - p64) * per32 <= sms) w.pairs64 = (int)p64;
    }
    return w;
}

namespace {

// State walk over pairs pair0 .. pair0 + n_pairs - 1 with value blocks of BV
// rows (D / BV CTAs per pair), reading the transforms in the workspace.
// With `pdl` the launch is a programmatic dependent launch behind the
// transform kernel: its CTAs load their state and first tiles while the
// transform grid finishes, and its workspace reads wait for that grid.
template <int D, int BV, bool NORM>
cudaError_t launch_walk_part(const Problem &p, const CUtensorMap &mq, const CUtensorMap &mk,
                             const uint8_t *zws, int pair0, int n_pairs, bool pdl,
                             cudaStream_t stream) {
    using CF = Cfg<D, BV>;
    CUtensorMap mv;
    if (!make_map(&mv, p.v, p.B, p.T, p.H, D, CF::BV)) return cudaErrorInvalidValue;
    static PerDeviceOnce attrs;
    const cudaError_t attr_err = attrs.run([] {
        return cudaFuncSetAttribute(chunked_kernel<D, BV, NORM>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_pairs * CF::NVB));
    cfg.blockDim = dim3(CF::NTH);
    cfg.dynamicSmemBytes = CF::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chunked_kernel<D, BV, NORM>, mq, mk, mv, p.g, p.beta,
                              p.state_in, p.state_out, p.out, zws, p.T, p.H, p.Hk, p.scale,
                              p.status, p.out_bf16, pair0);
}

// head_dim 256, and head_dim 128 with few pairs: the chunk transform for
// every chunk into the workspace, then the state walk reading it, in value
// blocks chosen by walk_split.
template <int D, bool NORM>
cudaError_t launch_d(const Problem &p, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    using ZC = ZCfg<D>;
    const int n_chunks = (p.T + C - 1) / C;
    const long long n_tasks = (long long)p.B * p.H * n_chunks;
    if (!workspace || ws_bytes < (size_t)n_tasks * Z_BYTES || n_tasks > INT_MAX)
        return cudaErrorInvalidValue;
    CUtensorMap mq, mk;
    if (!make_map(&mq, p.q, p.B, p.T, p.Hk, D, 64) || !make_map(&mk, p.k, p.B, p.T, p.Hk, D, 64))
        return cudaErrorInvalidValue;
    static PerDeviceOnce attrs;
    const cudaError_t attr_err = attrs.run([] {
        return cudaFuncSetAttribute(chunk_z_kernel<D, NORM>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, ZC::SMEM);
    });
    if (attr_err != cudaSuccess) return attr_err;
    uint8_t *zws = static_cast<uint8_t *>(workspace);
    const int sms = current_sm_count();
    const long long z_grid = std::min<long long>(n_tasks, 3LL * sms);
    chunk_z_kernel<D, NORM><<<(unsigned)z_grid, NT, ZC::SMEM, stream>>>(
        mq, mk, p.g, p.beta, zws, p.T, p.H, p.Hk, n_chunks, (int)n_tasks, p.status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const WalkSplit ws = walk_split(p.B * p.H, D, sms);
    if (ws.pairs64 > 0) {
        e = launch_walk_part<D, 64, NORM>(p, mq, mk, zws, 0, ws.pairs64, true, stream);
        if (e != cudaSuccess) return e;
    }
    if (ws.pairs64 < p.B * p.H)
        e = launch_walk_part<D, 32, NORM>(p, mq, mk, zws, ws.pairs64, p.B * p.H - ws.pairs64,
                                          ws.pairs64 == 0, stream);
    return e;
}

template <int D, bool NORM>
cudaError_t launch_ws(const Problem &p, cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, p.q, p.B, p.T, p.Hk, D, 64) ||
        !make_map(&mk, p.k, p.B, p.T, p.Hk, D, 64) ||
        !make_map(&mv, p.v, p.B, p.T, p.H, D, 64) ||
        !make_map_out(&mo, p.out, p.B, p.T, p.H, D, p.out_bf16))
        return cudaErrorInvalidValue;
    static PerDeviceOnce attrs;
    const cudaError_t attr_err = attrs.run([] {
        return cudaFuncSetAttribute(d128::chunked_d128_kernel<D, NORM>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, d128::SMEM);
    });
    if (attr_err != cudaSuccess) return attr_err;
    d128::chunked_d128_kernel<D, NORM><<<(unsigned)(p.B * p.H), d128::NTH, d128::SMEM, stream>>>(
        mq, mk, mv, mo, p.g, p.beta, p.state_in, p.state_out, p.out, p.T, p.H, p.Hk, p.scale,
        p.status, p.out_bf16);
    return cudaGetLastError();
}

// Self-test of the bounded waits: one CTA waits on an mbarrier that nothing
// ever arrives at, for at most `budget` SM clock cycles, and records
// GDN_ERR_TIMEOUT in the status word exactly as the chunked kernels do when
// one of their waits gives up.  The kernel then returns normally.
__global__ void wait_selftest_kernel(int *status, long long budget) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        ptx::mbar_init(&bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (!ptx::mbar_wait(&bar, 0, &abort_flag, budget)) {
        if (atomicExch(&abort_flag, 1) == 0) atomicExch(status, GDN_ERR_TIMEOUT);
    }
    __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(int *status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, 200000LL);
    return cudaGetLastError();
}

bool chunked_supports(int d) { return d == 64 || d == 128 || d == 256; }

// Below this many (sequence, head) pairs, head_dim 128 runs the two-kernel
// path (chunk transforms into the workspace, then a state walk with two
// value blocks per head): the fused kernel's one CTA per pair would leave
// most SMs idle.  Measured at 4096 tokens: 32 pairs 431 -> 325 us, 64 pairs
// 431 -> 394 us, 128 pairs 435 -> 764 us (fused -> two-kernel).
constexpr long long kD128SplitMaxPairs = 80;

bool d128_split(int B, int H) { return (long long)B * H < kD128SplitMaxPairs; }

// head_dim 64 (and 128 with many pairs) keep every chunk intermediate on
// chip; head_dim 256 (and 128 with few pairs) keep one 32 KB transform tile
// per (sequence, head, chunk) in the workspace.
size_t chunked_workspace_bytes(int B, int T, int H, int d, int) {
    if (B <= 0 || T <= 0 || H <= 0) return 0;
    if (d != 256 && !(d == 128 && d128_split(B, H))) return 0;
    const size_t n_chunks = ((size_t)T + C - 1) / C;
    return (size_t)B * (size_t)H * n_chunks * (size_t)Z_BYTES;
}

template <int D, bool NORM>
cudaError_t launch_walk(const Problem &p, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    return launch_d<D, NORM>(p, workspace, ws_bytes, stream);
}

template <bool NORM>
cudaError_t launch_chunked_t(const Problem &p, void *workspace, size_t ws_bytes,
                             cudaStream_t stream) {
    switch (p.d) {
        case 64: return launch_ws<64, NORM>(p, stream);
        case 128:
            return d128_split(p.B, p.H) ? launch_walk<128, NORM>(p, workspace, ws_bytes, stream)
                                        : launch_ws<128, NORM>(p, stream);
        case 256: return launch_walk<256, NORM>(p, workspace, ws_bytes, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_chunked(const Problem &p, void *workspace, size_t ws_bytes,
                           cudaStream_t stream) {
    if (p.dtype != GDN_DTYPE_BF16) return cudaErrorInvalidValue;
    return p.l2norm_qk ? launch_chunked_t<true>(p, workspace, ws_bytes, stream)
                       : launch_chunked_t<false>(p, workspace, ws_bytes, stream);
}

}  // namespace gdn
