// Decode attention (the flash_attn op of the "marcsun13/ggml-gated-delta-net"
// model card, section "flash_attn"): for every sequence b, query head h and
// query i,
//     out[b, i, h, :] = softmax_j(scale q[b,h,i] . k[b,hk,j] + mask[b,0,i,j]) v[b,hk,j,:]
// with hk = h / (n_heads / n_heads_kv): grouped-query attention is native, k
// and v carry n_heads_kv heads and are never expanded.  Only the vector
// (decode) shape is served: fewer than 20 queries per call.
//
// Decode is a stream over the cache: per key, a few rows (query heads of the
// group x queries) each take one dot product and one axpy over head_dim, so
// the kernel is bound by HBM once the per-key work is cheap.  Mapping on
// sm_103a:
//   * the R = (n_heads / n_heads_kv) * n_q rows of one kv head are cut into
//     row groups of RG rows; one thread-block cluster of CL <= 16 CTAs serves
//     (sequence, kv head, row block), and the cluster's CL x (warps per row
//     group) warps split the keys into contiguous ranges; CL grows when there
//     are few (sequence, kv head) pairs to fill the GPU with;
//   * a warp streams its keys through its own ring of shared memory (three
//     stages on the MMA path where they fit, else two) filled by asynchronous
//     copies (the next steps' k and v land while this one is computed; no
//     block barrier), and keeps its own online softmax (running max, sum of
//     exp, output slice) per row;
//   * 16-bit inputs (bf16, f16): per step of 16 keys a warp forms
//     S^T = K Q^T and O^T += V^T P^T with warp-level tensor-core MMAs
//     (m16n8k16, fp32 accumulators; 8 rows per warp as the N dimension):
//     k and v feed the MMAs straight from the stage, q waits in registers,
//     and the probabilities enter as hi + lo 16-bit pairs;
//   * fp32 inputs: each lane (head_dim/64 lanes per key) reads its key's k row
//     across the padded stage (one bank group per lane) against the CTA's
//     q rows, which are broadcast from shared memory; P V: each lane owns
//     head_dim/32 value columns and reads the step's probabilities as one
//     128-bit load per key; both accumulate with packed fp32 FMAs;
//   * at the end the warps of a CTA merge through shared memory and the CTAs
//     of the cluster through distributed shared memory, so no partial result
//     goes through global scratch.
// Accumulation is fp32; q, k and v enter exactly (upcast, or as 16-bit MMA
// operands) and the MMA path's probabilities as hi + lo pairs (upstream
// accumulates in f16; that is its kernel's choice, not part of the operation).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace attn {
namespace {

constexpr int MAX_CLUSTER = 16; // largest cluster the merge handles (non-portable size)

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {   // at most N most recent groups pending
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of `p` (a shared-memory pointer of this CTA) in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(const void *p, int rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// Reads of peers' partials, only between the two cluster barriers: volatile
// keeps them after the first barrier (volatile asm keeps its order), and
// without a memory clobber they can still be issued back to back.
__device__ __forceinline__ float ld_peer(uint32_t addr) {
    float x;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x) : "r"(addr));
    return x;
}

// A lane's SL consecutive fp32 elements of one row (SL = head_dim / 32), raw
// (packed-FMA path).
template <typename Tin, int SL>
struct Slice {
    static constexpr int BYTES = SL * (int)sizeof(Tin);
    static constexpr int WORDS = BYTES / 4;
    uint32_t w[WORDS];
};
// from shared memory
template <typename Tin, int SL>
__device__ __forceinline__ void ld_slice(Slice<Tin, SL> &s, const Tin *p) {
    constexpr int B = Slice<Tin, SL>::BYTES;
    if constexpr (B == 8) {
        const uint2 a = *reinterpret_cast<const uint2 *>(p);
        s.w[0] = a.x; s.w[1] = a.y;
    } else {
        static_assert(B % 16 == 0, "slice of 2, 4 or 8 floats");
#pragma unroll
        for (int i = 0; i < B / 16; ++i) {
            const uint4 a = *(reinterpret_cast<const uint4 *>(p) + i);
            s.w[4 * i] = a.x; s.w[4 * i + 1] = a.y; s.w[4 * i + 2] = a.z; s.w[4 * i + 3] = a.w;
        }
    }
}
template <int SL>
__device__ __forceinline__ void unpack(const Slice<float, SL> &s, float (&x)[SL]) {
#pragma unroll
    for (int i = 0; i < SL; ++i) x[i] = __uint_as_float(s.w[i]);
}
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

// Packed fp32 FMA on two lanes of a 64-bit register pair (sm_100 family):
// d = a * b + c element by element, each rounded as fmaf rounds it.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// 16-byte copy that writes zeros and reads nothing (source size 0); `src` is
// still a valid address of the range.
__device__ __forceinline__ void cp_async16_zero(void *dst, const void *src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(0)
                 : "memory");
}

// Warp-level tensor-core pieces of the 16-bit path.  ldmatrix hands every
// lane its part of four 8 x 8 tiles of 16-bit elements, lanes 8i .. 8i + 7
// naming the 16-byte rows of tile i (.trans: the tiles transposed);
// mma.sync m16n8k16 (A row-major 16 x 16, B column-major 16 x 8) accumulates
// in fp32.  Fragment of lane (g = lane / 4, t = lane % 4): A rows g, g + 8 and
// columns 2t, 2t + 1, 2t + 8, 2t + 9; B columns (n) g and rows (k) 2t, 2t + 1,
// 2t + 8, 2t + 9; C rows g, g + 8 and columns 2t, 2t + 1.
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void *p) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a) : "memory");
}
__device__ __forceinline__ void ldsm4_t(uint32_t (&r)[4], const void *p) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a) : "memory");
}
template <typename Tin>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value)
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    else
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// x0, x1 (fp32) as two 16-bit pairs, hi = (x0, x1) rounded and lo = the
// rounded remainders, so hi + lo carries about 16 significant bits (the
// first element in the low half, as the MMA fragments order them)
template <typename Tin>
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
        const float2 f = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - f.x, x1 - f.y);
        hi = *reinterpret_cast<const uint32_t *>(&h);
        lo = *reinterpret_cast<const uint32_t *>(&l);
    } else {
        const __half2 h = __floats2half2_rn(x0, x1);
        const float2 f = __half22float2(h);
        const __half2 l = __floats2half2_rn(x0 - f.x, x1 - f.y);
        hi = *reinterpret_cast<const uint32_t *>(&h);
        lo = *reinterpret_cast<const uint32_t *>(&l);
    }
}
constexpr int kPTS = 20;          // row stride (floats) of a warp's probabilities, [row][key]

// Scores are kept in log2 units (q pre-scaled by scale * log2 e, the mask by
// log2 e), so every exponential of the softmax is a hardware 2^x; the
// softmax is unchanged by the base.  Results below the fp32 normal range
// flush to zero.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 8 consecutive elements of a row in shared memory, as fp32
__device__ __forceinline__ void lds8(const float *p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
// 8 consecutive fp32 elements of q in global memory (packed-FMA path)
__device__ __forceinline__ void ldg8(const float *p, float (&x)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Geometry for key / query width DK, value width DV and input type Tin.
// 16-bit inputs (MMA): a step is NKS = 16 keys (the M of S^T = K Q^T and the
//   K of O^T += V^T P^T) and a warp carries RG = 8 rows (their N); k and v
//   rows are both padded by 16 bytes, so the 8 rows of an ldmatrix tile fall
//   on distinct banks.
// fp32 inputs:
//   scores: KPL = max(DK, DV)/64 lanes share a key (each a DQ = DK/KPL-element
//           part of its row), so a step holds NKS = 32/KPL keys, one per lane
//           group (wide value rows keep the step, and the ring, small);
//   P V:    every lane owns SL = DV/32 consecutive value columns;
//   a warp carries RG = 4 rows (query head of the group x query).
// A warp's ring holds ST steps of NKS keys of k (rows padded by 16 bytes, so
// that lanes reading different rows hit different banks) and v.
template <int DK, int DV, typename Tin> struct Geo {
    static constexpr int ELT = (int)sizeof(Tin);
    static constexpr bool MMA = ELT == 2;
    static constexpr int KPL = MMA ? 1 : (DK > DV ? DK : DV) / 64;
    static constexpr int NKS = MMA ? 16 : 32 / KPL;
    static constexpr int DQ = DK / KPL;
    static constexpr int SL = DV / 32;
    static constexpr int RG = MMA ? 8 : 4;
    static constexpr int KST = DK * ELT + 16;
    static constexpr int VST = DV * ELT + (MMA ? 16 : 0);
    static constexpr int STEP = NKS * (KST + VST);
    // warps per CTA: 8 while their rings take at most 200 KB
    static constexpr int NW = ELT == 4 ? 4 : (8 * 2 * STEP <= 200 * 1024 ? 8 : 4);
    // ring stages per warp: three on the MMA path where they fit (its steps
    // are short, so more copies must be in flight), else two
    static constexpr int ST = MMA && NW * 3 * STEP <= 212 * 1024 ? 3 : 2;
    static constexpr int NTHR = NW * 32;
    static constexpr int RING = NW * ST * STEP;
    // after the key loop the ring is reused for the merge buffers
    static constexpr int WO = 0;                                  // [NW][RG][DV] fp32
    static constexpr int CO = WO + NW * RG * DV * 4;              // [NW*RG][DV] fp32
    static constexpr int MERGE = CO + NW * RG * DV * 4;
    static constexpr int QOFF = RING > MERGE ? RING : MERGE;      // the CTA's q rows, fp32
    static constexpr int SMEM = QOFF + (MMA ? 0 : NW * RG * DK * 4);
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(KST % 16 == 0 && STEP % 16 == 0 && QOFF % 16 == 0, "alignment");
    static_assert(MMA || (DQ % 8 == 0 && KPL * NKS == 32), "score split");
    static_assert(!MMA || (DK % 16 == 0 && DV % 16 == 0), "MMA tiles");
    static_assert((NKS * (DK * ELT / 16)) % 32 == 0 && (NKS * (DV * ELT / 16)) % 32 == 0,
                  "whole copies per lane");
};

// Small per-CTA state outside the ring.
template <int NW, int RG, int NKS, bool MMA>
struct SmallSmem {
    float wm[NW][RG], wl[NW][RG];                     // each warp's partial max (then weight), sum
    float cm[NW * RG], cl[NW * RG];                   // the CTA's partial per local row
    float pw[NW * RG][MAX_CLUSTER];                   // cluster merge: weight of each CTA per row
    float pl[NW * RG];                                // cluster merge: total sum of exp per row
    float p[NW][MMA ? 1 : NKS][RG];                   // a step's probabilities, [key][row]
    float pt[NW][MMA ? RG * kPTS : 1];                // ... on the MMA path, [row][key]
};

template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(Geo<DK, DV, Tin>::NTHR, 1)
attn_decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                   const Tin *__restrict__ v, const Tin *__restrict__ mask,
                   float *__restrict__ out, int H, int Hkv, int n_q, int n_kv, int n_rb, int n_rgc,
                   int CL, float scale)
{
    using G = Geo<DK, DV, Tin>;
    constexpr int SL = G::SL, RG = G::RG, NW = G::NW, ST = G::ST, NTHR = G::NTHR;
    constexpr int NKS = G::NKS, DQ = G::DQ;
    extern __shared__ __align__(16) uint8_t ring[];
    __shared__ __align__(16) SmallSmem<NW, RG, NKS, G::MMA> sm;
    static_assert(G::SMEM + sizeof(sm) <= 227 * 1024, "shared memory (dynamic + static)");
    float (*wo)[RG][DV] = reinterpret_cast<float (*)[RG][DV]>(ring + G::WO);
    float (*co)[DV] = reinterpret_cast<float (*)[DV]>(ring + G::CO);
    float *sQ = reinterpret_cast<float *>(ring + G::QOFF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t rank_u;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank_u));
    const int rank = (int)rank_u;                     // 0 .. CL-1 (cluster dims CL x 1 x 1)
    const int unit = (int)(blockIdx.x / (unsigned)CL);
    const int rb = unit % n_rb;
    const int bhk = unit / n_rb;
    const int b = bhk / Hkv, hk = bhk - b * Hkv;
    const int rep = H / Hkv;
    const int R = rep * n_q;                          // rows (query head, query) of this kv head
    const int n_ksc = NW / n_rgc;                     // warps per row group in a CTA
    const int rgc = warp % n_rgc;                     // this warp's row group in the CTA
    const int ksw = warp / n_rgc;                     // this warp's key split in the CTA
    const int rows_cta = n_rgc * RG;
    const int rbase = rb * rows_cta;
    const int r0 = rbase + rgc * RG;                  // first row of this warp
    const int nr = max(0, min(RG, R - r0));

    // key range of this warp: split s of S = CL * n_ksc, in steps of NKS keys
    const int S = CL * n_ksc;
    const int s = rank * n_ksc + ksw;
    const int n_steps_all = (n_kv + NKS - 1) / NKS;
    const int sps = (n_steps_all + S - 1) / S;
    const int kb = min(n_kv, s * sps * NKS);
    const int ke = min(n_kv, kb + sps * NKS);
    const int n_steps = nr > 0 ? (ke - kb + NKS - 1) / NKS : 0;

    const Tin *kg = k + (size_t)(b * Hkv + hk) * n_kv * DK;
    const Tin *vg = v + (size_t)(b * Hkv + hk) * n_kv * DV;
    uint8_t *wring = ring + warp * ST * G::STEP;
    // stage `st` <- keys kb + NKS*step ..: k rows (padded), then v rows; rows
    // past the range are not copied (their scores are masked, their v rows
    // skipped) or, on the MMA path, zero-filled (an MMA cannot skip a key)
    auto issue = [&](int step, int st) {
        if (step < n_steps) {
            const int j0 = kb + step * NKS;
            const int nk = min(NKS, ke - j0);
            constexpr int CPK = DK * G::ELT / 16;     // 16-byte copies per k row
            constexpr int CPV = DV * G::ELT / 16;     // ... per v row
            uint8_t *dk = wring + st * G::STEP;
            uint8_t *dv = dk + NKS * G::KST;
            const uint8_t *sk = reinterpret_cast<const uint8_t *>(kg + (size_t)j0 * DK);
            const uint8_t *sv = reinterpret_cast<const uint8_t *>(vg + (size_t)j0 * DV);
            // copy i of this lane: piece c = lane + 32 i of the stage, row c / CP,
            // 16-byte column c % CP; unrolled, so only the lane's first row and
            // column are computed at run time
#pragma unroll
            for (int i = 0; i < NKS * CPK / 32; ++i) {
                const int g = CPK <= 32 ? lane / CPK + i * (32 / CPK) : i / (CPK / 32);
                const int x = CPK <= 32 ? lane % CPK : lane + 32 * (i % (CPK / 32));
                if (g < nk) cp_async16(dk + g * G::KST + x * 16, sk + (size_t)g * (DK * G::ELT) + x * 16);
                else if constexpr (G::MMA) cp_async16_zero(dk + g * G::KST + x * 16, sk + x * 16);
            }
#pragma unroll
            for (int i = 0; i < NKS * CPV / 32; ++i) {
                const int g = CPV <= 32 ? lane / CPV + i * (32 / CPV) : i / (CPV / 32);
                const int x = CPV <= 32 ? lane % CPV : lane + 32 * (i % (CPV / 32));
                if (g < nk) cp_async16(dv + g * G::VST + x * 16, sv + (size_t)g * (DV * G::ELT) + x * 16);
                else if constexpr (G::MMA) cp_async16_zero(dv + g * G::VST + x * 16, sv + x * 16);
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < ST - 1; ++i) issue(i, i);

    if constexpr (G::MMA) {
        // Tensor-core path.  Per step of NKS = 16 keys a warp forms
        //   S^T  = K Q^T     (M = 16 keys, N = 8 rows, K = DK; A = the k rows
        //                     of the stage, B = q in registers)
        //   O^T += V^T P^T   (per 16 value columns: M = 16, N = 8 rows,
        //                     K = 16 keys; A = the v rows transposed by
        //                     ldmatrix, B = the probabilities as hi + lo)
        // Lane (gi, ti) holds the S^T and O^T entries of rows 2ti and 2ti + 1
        // of the warp, and keeps the online softmax of those two rows.
        const int gi = lane >> 2, ti = lane & 3;
        const int rho0 = 2 * ti;
        const float sl = scale * kLog2e;
        // q as B fragments: row gi of the warp, columns 16s + 2ti (+1) and
        // 16s + 8 + 2ti (+1); rows past the valid ones are zeros
        uint32_t qf[DK / 16][2];
        {
            const bool ok = gi < nr;
            const uint32_t *qr = reinterpret_cast<const uint32_t *>(
                q + ((size_t)(b * H + hk * rep) * n_q + (ok ? r0 + gi : 0)) * DK);
#pragma unroll
            for (int s2 = 0; s2 < DK / 16; ++s2) {
                qf[s2][0] = ok ? __ldg(qr + s2 * 8 + ti) : 0u;
                qf[s2][1] = ok ? __ldg(qr + s2 * 8 + 4 + ti) : 0u;
            }
        }
        float oacc[DV / 16][4];
#pragma unroll
        for (int mt = 0; mt < DV / 16; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[mt][e] = 0.f;
        float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};
        float *pt = sm.pt[warp];
        // ldmatrix row addresses: k tiles (keys lane & 15, 16-byte half lane >> 4),
        // v tiles transposed (keys (lane & 7) + 8 (lane >> 4), half (lane >> 3) & 1)
        const int koff = (lane & 15) * G::KST + (lane >> 4) * 16;
        const int voff = ((lane & 7) + ((lane >> 4) << 3)) * G::VST + ((lane >> 3) & 1) * 16;
        for (int step = 0; step < n_steps; ++step) {
            cp_async_wait<ST - 2>();                  // this step's copies (own lane) landed
            __syncwarp();                             // ... and every lane's
            issue(step + ST - 1, (step + ST - 1) % ST);
            const int j0 = kb + step * NKS;
            const int nk = min(NKS, ke - j0);
            const uint8_t *sk = wring + (step % ST) * G::STEP;
            const uint8_t *sv = sk + NKS * G::KST;

            // ---- S^T = K Q^T, two accumulators (even / odd column blocks)
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s2 = 0; s2 < DK / 16; ++s2) {
                uint32_t a[4];
                ldsm4(a, sk + koff + s2 * 32);
                if (s2 & 1) mma16816<Tin>(sb, a, qf[s2][0], qf[s2][1]);
                else        mma16816<Tin>(sa, a, qf[s2][0], qf[s2][1]);
            }
            // entry e: key gi + 8 (e >> 1), row rho0 + (e & 1); scores in log2 units
            float sc[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = gi + (e >> 1) * 8, row = rho0 + (e & 1);
                float x = (sa[e] + sb[e]) * sl;
                if (key < nk && row < nr) {
                    if (mask) {
                        const int i = (r0 + row) % n_q;
                        x = fmaf(to_f32(mask[((size_t)b * n_q + i) * n_kv + j0 + key]), kLog2e, x);
                    }
                } else {
                    x = -INFINITY;
                }
                sc[e] = x;
            }
            // ---- online softmax of rows rho0, rho0 + 1 (the step's 16 keys
            //      sit on the 8 lanes of equal ti, two per lane)
            float mx[2] = {fmaxf(sc[0], sc[2]), fmaxf(sc[1], sc[3])};
#pragma unroll
            for (int off = 4; off < 32; off <<= 1)
#pragma unroll
                for (int r = 0; r < 2; ++r) mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], off));
            float cf[2], pv[4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float m_new = fmaxf(mr[r], mx[r]);
                const bool none = (m_new == -INFINITY);
                cf[r] = none ? 1.f : exp2_approx(mr[r] - m_new);
                pv[r] = none ? 0.f : exp2_approx(sc[r] - m_new);
                pv[r + 2] = none ? 0.f : exp2_approx(sc[r + 2] - m_new);
                lr[r] = fmaf(lr[r], cf[r], pv[r] + pv[r + 2]);   // this lane's keys only
                mr[r] = m_new;
            }
            if (__any_sync(0xffffffffu, cf[0] != 1.f || cf[1] != 1.f)) {
#pragma unroll
                for (int mt = 0; mt < DV / 16; ++mt) {
                    oacc[mt][0] *= cf[0]; oacc[mt][1] *= cf[1];
                    oacc[mt][2] *= cf[0]; oacc[mt][3] *= cf[1];
                }
            }
            // ---- probabilities to [row][key], read back as B fragments:
            //      keys 2ti, 2ti + 1 and 2ti + 8, 2ti + 9 of row gi
            pt[rho0 * kPTS + gi] = pv[0];
            pt[(rho0 + 1) * kPTS + gi] = pv[1];
            pt[rho0 * kPTS + gi + 8] = pv[2];
            pt[(rho0 + 1) * kPTS + gi + 8] = pv[3];
            __syncwarp();
            const float2 u = *reinterpret_cast<const float2 *>(pt + gi * kPTS + 2 * ti);
            const float2 w = *reinterpret_cast<const float2 *>(pt + gi * kPTS + 2 * ti + 8);
            uint32_t bh0, bl0, bh1, bl1;
            split2<Tin>(u.x, u.y, bh0, bl0);
            split2<Tin>(w.x, w.y, bh1, bl1);
            // ---- O^T += V^T P^T (keys past the range: zero rows, zero weights)
#pragma unroll
            for (int mt = 0; mt < DV / 16; ++mt) {
                uint32_t a[4];
                ldsm4_t(a, sv + voff + mt * 32);
                mma16816<Tin>(oacc[mt], a, bh0, bh1);
                mma16816<Tin>(oacc[mt], a, bl0, bl1);
            }
            __syncwarp();                             // stage and probabilities consumed
        }
        // each row's sum over the 8 lanes that hold its keys
#pragma unroll
        for (int off = 4; off < 32; off <<= 1)
#pragma unroll
            for (int r = 0; r < 2; ++r) lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], off);
        cp_async_wait<0>();
        __syncthreads();                              // every warp is done with the ring

        // ---- this warp's partials for the merge below
        if (gi == 0) {
            sm.wm[warp][rho0] = mr[0];
            sm.wm[warp][rho0 + 1] = mr[1];
            sm.wl[warp][rho0] = lr[0];
            sm.wl[warp][rho0 + 1] = lr[1];
        }
#pragma unroll
        for (int mt = 0; mt < DV / 16; ++mt) {
            wo[warp][rho0][mt * 16 + gi] = oacc[mt][0];
            wo[warp][rho0 + 1][mt * 16 + gi] = oacc[mt][1];
            wo[warp][rho0][mt * 16 + gi + 8] = oacc[mt][2];
            wo[warp][rho0 + 1][mt * 16 + gi + 8] = oacc[mt][3];
        }
    } else {
        // the CTA's rows of q, scaled by scale * log2 e, fp32 (rows past R: zeros); rows rbase + lr
        // are consecutive in q: head hk*rep + row / n_q, query row % n_q
        for (int i = tid; i < rows_cta * (DK / 8); i += NTHR) {
            const int lr = i / (DK / 8), c = i - lr * (DK / 8);
            const int rg = rbase + lr;
            float x[8];
            if (rg < R) {
                ldg8(q + ((size_t)(b * H + hk * rep) * n_q + rg) * DK + c * 8, x);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = 0.f;
            }
            float4 *dst = reinterpret_cast<float4 *>(sQ + lr * DK + c * 8);
            const float sl = scale * kLog2e;
            dst[0] = make_float4(sl * x[0], sl * x[1], sl * x[2], sl * x[3]);
            dst[1] = make_float4(sl * x[4], sl * x[5], sl * x[6], sl * x[7]);
        }
        __syncthreads();

        float m[RG], l[RG];
        float2 acc[RG][SL / 2];
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
#pragma unroll
            for (int e = 0; e < SL / 2; ++e) acc[r][e] = make_float2(0.f, 0.f);
        }
        const int key = lane % NKS, part = lane / NKS;    // score pass: this lane's key and row part
        const float *qw = sQ + (rgc * RG) * DK + part * DQ;

        for (int step = 0; step < n_steps; ++step) {
            cp_async_wait<ST - 2>();                      // this step's copies (own lane) landed
            __syncwarp();                                 // ... and every lane's
            // refill the stage the previous step used (every lane passed the
            // __syncwarp after reading it) while this step is computed
            issue(step + ST - 1, (step + ST - 1) % ST);
            const int j0 = kb + step * NKS;
            const int nk = min(NKS, ke - j0);
            const uint8_t *sk = wring + (step % ST) * G::STEP;
            const Tin *sv = reinterpret_cast<const Tin *>(sk + NKS * G::KST);

            // ---- scores: q . k over this lane's part of its key's row
            float2 a2[RG];
#pragma unroll
            for (int r = 0; r < RG; ++r) a2[r] = make_float2(0.f, 0.f);
            const Tin *krow = reinterpret_cast<const Tin *>(sk + key * G::KST) + part * DQ;
#pragma unroll 4
            for (int c = 0; c < DQ / 8; ++c) {
                float kx[8];
                lds8(krow + c * 8, kx);
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    float qx[8];
                    lds8(qw + r * DK + c * 8, qx);
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        a2[r] = ffma2(make_float2(qx[e], qx[e + 1]), make_float2(kx[e], kx[e + 1]),
                                      a2[r]);
                }
            }
            // ---- online softmax over the step's keys, all RG rows side by side
            //      (rows past the warp's valid rows are masked out, not branched
            //      around, so each reduction level issues RG independent shuffles)
            float sc[RG];
#pragma unroll
            for (int r = 0; r < RG; ++r) sc[r] = a2[r].x + a2[r].y;
#pragma unroll
            for (int off = NKS; off < 32; off <<= 1)
#pragma unroll
                for (int r = 0; r < RG; ++r) sc[r] += __shfl_xor_sync(0xffffffffu, sc[r], off);
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                if (r < nr && key < nk) {
                    if (mask) {
                        const int i = (r0 + r) % n_q;
                        sc[r] = fmaf(to_f32(mask[((size_t)b * n_q + i) * n_kv + j0 + key]), kLog2e,
                                     sc[r]);
                    }
                } else {
                    sc[r] = -INFINITY;
                }
            }
            float gm[RG];
#pragma unroll
            for (int r = 0; r < RG; ++r) gm[r] = sc[r];
#pragma unroll
            for (int off = 1; off < NKS; off <<= 1)
#pragma unroll
                for (int r = 0; r < RG; ++r) gm[r] = fmaxf(gm[r], __shfl_xor_sync(0xffffffffu, gm[r], off));
            float pv[RG], ps[RG], cf[RG];
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                const float m_new = fmaxf(m[r], gm[r]);
                const bool none = (m_new == -INFINITY);
                pv[r] = none ? 0.f : exp2_approx(sc[r] - m_new);
                cf[r] = none ? 1.f : exp2_approx(m[r] - m_new);
                m[r] = m_new;
                ps[r] = pv[r];
            }
#pragma unroll
            for (int off = 1; off < NKS; off <<= 1)
#pragma unroll
                for (int r = 0; r < RG; ++r) ps[r] += __shfl_xor_sync(0xffffffffu, ps[r], off);
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                l[r] = fmaf(l[r], cf[r], ps[r]);
#pragma unroll
                for (int e = 0; e < SL / 2; ++e)
                    acc[r][e] = make_float2(acc[r][e].x * cf[r], acc[r][e].y * cf[r]);
            }
            static_assert(RG == 4, "one 128-bit store of the probabilities per key");
            if (part == 0)
                *reinterpret_cast<float4 *>(&sm.p[warp][key][0]) = make_float4(pv[0], pv[1], pv[2], pv[3]);
            __syncwarp();
            // ---- P V on this lane's value columns (keys past the range skipped:
            //      their stage rows hold stale data)
#pragma unroll 2
            for (int g = 0; g < nk; ++g) {
                Slice<Tin, SL> vr;
                ld_slice(vr, sv + g * DV + lane * SL);
                float vx[SL];
                unpack(vr, vx);
                const float4 p4 = *reinterpret_cast<const float4 *>(&sm.p[warp][g][0]);
                const float pr[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                for (int r = 0; r < RG; ++r)
#pragma unroll
                    for (int e = 0; e < SL / 2; ++e)
                        acc[r][e] = ffma2(make_float2(pr[r], pr[r]), make_float2(vx[2 * e], vx[2 * e + 1]),
                                          acc[r][e]);
            }
            __syncwarp();                                 // stage and probabilities consumed
        }
        cp_async_wait<0>();
        __syncthreads();                                  // every warp is done with the ring

        // ---- merge the warps of this CTA (same row group, different keys).  The
        //      weights exp(m_w - M) depend only on the row: one thread per row
        //      computes them (in place of the maxima) and the row's M and L.
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            if (lane == 0) { sm.wm[warp][r] = m[r]; sm.wl[warp][r] = l[r]; }
#pragma unroll
            for (int e = 0; e < SL / 2; ++e) {
                wo[warp][r][lane * SL + 2 * e] = acc[r][e].x;
                wo[warp][r][lane * SL + 2 * e + 1] = acc[r][e].y;
            }
        }
    }
    __syncthreads();
    if (tid < rows_cta) {                             // local row lr = tid: group g, row r
        const int g = tid / RG, r = tid - g * RG;
        float M = -INFINITY;
        for (int w = g; w < NW; w += n_rgc) M = fmaxf(M, sm.wm[w][r]);
        float L = 0.f;
        for (int w = g; w < NW; w += n_rgc) {
            const float mw = sm.wm[w][r];
            const float wt = (M == -INFINITY || mw == -INFINITY) ? 0.f : exp2_approx(mw - M);
            L = fmaf(wt, sm.wl[w][r], L);
            sm.wm[w][r] = wt;                         // each warp belongs to one row group
        }
        sm.cm[tid] = M;
        sm.cl[tid] = L;
    }
    __syncthreads();
    for (int it = tid; it < rows_cta * DV; it += NTHR) {
        const int lr = it / DV, col = it - lr * DV;
        const int g = lr / RG, r = lr - g * RG;
        float o = 0.f;
        for (int w = g; w < NW; w += n_rgc) o = fmaf(sm.wm[w][r], wo[w][r][col], o);
        co[lr][col] = o;
    }
    // ---- merge the CTAs of the cluster (same rows, different keys): per row,
    //      each CTA's weight once, then the weighted sum per column
    cluster_sync();
    const int nr_cta = max(0, min(rows_cta, R - rbase));
    if (tid < nr_cta) {
        float mk[MAX_CLUSTER];
        float M = -INFINITY;
#pragma unroll
        for (int pr = 0; pr < MAX_CLUSTER; ++pr) {
            mk[pr] = pr < CL ? ld_peer(peer_addr(&sm.cm[tid], pr)) : -INFINITY;
            M = fmaxf(M, mk[pr]);
        }
        float L = 0.f;
#pragma unroll
        for (int pr = 0; pr < MAX_CLUSTER; ++pr) {
            float wt = 0.f;
            if (pr < CL && M != -INFINITY && mk[pr] != -INFINITY) {
                wt = exp2_approx(mk[pr] - M);
                L = fmaf(wt, ld_peer(peer_addr(&sm.cl[tid], pr)), L);
            }
            sm.pw[tid][pr] = wt;
        }
        sm.pl[tid] = L;
    }
    __syncthreads();
    for (int it = rank * NTHR + tid; it < nr_cta * DV; it += CL * NTHR) {
        const int lr = it / DV, col = it - lr * DV;
        float o = 0.f;
#pragma unroll
        for (int pr = 0; pr < MAX_CLUSTER; ++pr) {
            const float wt = sm.pw[lr][pr];
            if (pr < CL && wt != 0.f) o = fmaf(wt, ld_peer(peer_addr(&co[lr][col], pr)), o);
        }
        const float L = sm.pl[lr];
        const int rg = rbase + lr;
        const int h = hk * rep + rg / n_q, i = rg % n_q;
        out[(((size_t)b * n_q + i) * H + h) * DV + col] = (L > 0.f) ? o / L : 0.f;
    }
    cluster_sync();                                   // peers are done reading this CTA
}

struct AttnProblem {
    const void *q, *k, *v, *mask;
    float *out;
    int B, H, Hkv, n_q, n_kv, dk, dv;
    float scale;
};

template <int DK, int DV, typename Tin>
cudaError_t launch(const AttnProblem &p, cudaStream_t stream) {
    using G = Geo<DK, DV, Tin>;
    constexpr int RG = G::RG, NWARP = G::NW;
    const int rep = p.H / p.Hkv;
    const long long R = (long long)rep * p.n_q;
    // row groups per CTA: enough for the rows, a power of two dividing the warps
    int n_rgc = 1;
    while (n_rgc < NWARP && (long long)n_rgc * RG < R) n_rgc *= 2;
    const int n_ksc = NWARP / n_rgc;
    const int n_rb = (int)((R + (long long)n_rgc * RG - 1) / ((long long)n_rgc * RG));
    // one-time set-up per device: shared memory size, clusters beyond the
    // portable 8, and the largest cluster this kernel can actually be given
    static PerDeviceOnce setup;
    static int max_cl_of[kMaxDevices];
    const cudaError_t attr_err = setup.run([] {
        const int dev = current_device();
        max_cl_of[dev] = 8;
        cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<DK, DV, Tin>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
        if (e != cudaSuccess) return e;
        if (cudaFuncSetAttribute(attn_decode_kernel<DK, DV, Tin>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(MAX_CLUSTER);
            q.blockDim = dim3(G::NTHR);
            q.dynamicSmemBytes = G::SMEM;
            int n = 0;
            if (cudaOccupancyMaxPotentialClusterSize(&n, attn_decode_kernel<DK, DV, Tin>, &q) ==
                    cudaSuccess && n >= 8)
                max_cl_of[dev] = n < MAX_CLUSTER ? n : MAX_CLUSTER;
        }
        (void)cudaGetLastError();                    // a refused query leaves the portable 8
        return cudaSuccess;
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int max_cl = max_cl_of[current_device()];
    // CTAs per cluster: enough clusters x CTAs for about four waves of the GPU
    // (one CTA per SM; a partial last wave then costs little), but no more
    // CTAs than give every warp one step of keys.  A short or single-sequence
    // cache is spread over many SMs; a large batch keeps few CTAs per
    // (sequence, kv head, row block) and long key ranges per warp.
    const long long units = (long long)p.B * p.Hkv * n_rb;
    const long long fill = (4LL * current_sm_count() + units - 1) / units;
    const long long per_cta = (long long)n_ksc * G::NKS;
    const long long by_keys = (p.n_kv + per_cta - 1) / per_cta;
    long long cl = fill < by_keys ? fill : by_keys;
    if (cl > max_cl) cl = max_cl;
    if (cl < 1) cl = 1;
    const int CL = (int)cl;
    const long long blocks = units * CL;
    if (blocks > INT_MAX) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(G::NTHR);
    cfg.dynamicSmemBytes = G::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, attn_decode_kernel<DK, DV, Tin>, static_cast<const Tin *>(p.q),
                              static_cast<const Tin *>(p.k), static_cast<const Tin *>(p.v),
                              static_cast<const Tin *>(p.mask), p.out, p.H, p.Hkv, p.n_q, p.n_kv,
                              n_rb, n_rgc, CL, p.scale);
}

template <int DK, typename Tin>
cudaError_t launch_dv(const AttnProblem &p, cudaStream_t stream) {
    switch (p.dv) {
        case 64: return launch<DK, 64, Tin>(p, stream);
        case 128: return launch<DK, 128, Tin>(p, stream);
        case 256: return launch<DK, 256, Tin>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <typename Tin>
cudaError_t launch_dtype(const AttnProblem &p, cudaStream_t stream) {
    switch (p.dk) {
        case 64: return launch_dv<64, Tin>(p, stream);
        case 128: return launch_dv<128, Tin>(p, stream);
        case 256: return launch_dv<256, Tin>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

constexpr int kMaxQueries = 19;   // the vector (decode) variant: fewer than 20 queries

// key / query and value widths are independent: each of 64, 128 or 256
bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }
bool head_dims_ok(int dk, int dv) { return head_dim_ok(dk) && head_dim_ok(dv); }

}  // namespace
}  // namespace attn
}  // namespace gdn

extern "C" {

int gdn_flash_attn_supports(int n_q, int head_dim_k, int head_dim_v) {
    return (n_q >= 1 && n_q <= gdn::attn::kMaxQueries &&
            gdn::attn::head_dims_ok(head_dim_k, head_dim_v)) ? 1 : 0;
}

int gdn_flash_attn(const void *q, const void *k, const void *v, const void *mask, float *out,
                   int n_seqs, int n_heads, int n_heads_kv, int n_q, int n_kv, int head_dim_k,
                   int head_dim_v, float scale, int dtype, gdn_stream_t stream) {
    using namespace gdn::host;
    if (n_seqs < 0 || n_heads < 0 || n_heads_kv < 0 || n_q < 0 || n_kv < 0) return GDN_ERR_ARG;
    if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F16)
        return GDN_ERR_ARG;
    if (!gdn::attn::head_dims_ok(head_dim_k, head_dim_v)) return GDN_ERR_HEADDIM;
    if (n_q > gdn::attn::kMaxQueries) return GDN_ERR_SHAPE;
    if (n_heads > 0 && (n_heads_kv < 1 || n_heads % n_heads_kv != 0)) return GDN_ERR_ARG;
    if (!std::isfinite(scale)) return GDN_ERR_ARG;
    const unsigned long long elt = dtype == GDN_DTYPE_F32 ? 4 : 2;
    const unsigned long long dk = (unsigned long long)head_dim_k;
    const unsigned long long dv = (unsigned long long)head_dim_v;
    unsigned long long nq_rows, kv_rows, mask_n, q_bytes, k_bytes, v_bytes, mask_bytes, out_bytes;
    if (!mul_ok((unsigned long long)n_seqs * (unsigned long long)n_heads, (unsigned long long)n_q,
                &nq_rows) ||
        !mul_ok((unsigned long long)n_seqs * (unsigned long long)n_heads_kv,
                (unsigned long long)n_kv, &kv_rows) ||
        !mul_ok((unsigned long long)n_seqs * (unsigned long long)n_q, (unsigned long long)n_kv,
                &mask_n))
        return GDN_ERR_ARG;
    unsigned long long q_elems, out_elems, k_elems, v_elems;
    if (!mul_ok(nq_rows, dk, &q_elems) || !mul_ok(nq_rows, dv, &out_elems) ||
        !mul_ok(kv_rows, dk, &k_elems) || !mul_ok(kv_rows, dv, &v_elems) ||
        !span_bytes(q_elems, elt, &q_bytes) || !span_bytes(k_elems, elt, &k_bytes) ||
        !span_bytes(v_elems, elt, &v_bytes) || !span_bytes(mask_n, elt, &mask_bytes) ||
        !span_bytes(out_elems, 4, &out_bytes))
        return GDN_ERR_ARG;
    if (nq_rows == 0) return GDN_OK;                  // no queries: nothing to do
    if (!q || !out || (kv_rows > 0 && (!k || !v))) return GDN_ERR_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || (k && !aligned(k, 16)) || (v && !aligned(v, 16)) ||
        (mask && !aligned(mask, elt)))
        return GDN_ERR_ALIGN;
    const Range ro = range_of(out, out_bytes);
    for (Range in : {range_of(q, q_bytes), range_of(k, k_bytes), range_of(v, v_bytes),
                     range_of(mask, mask ? mask_bytes : 0)})
        if (overlap(ro, in)) return GDN_ERR_ALIAS;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (n_kv == 0)   // empty cache: every output row is zero
        return cudaMemsetAsync(out, 0, out_bytes, st) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    const gdn::attn::AttnProblem p{q, k, v, mask, out, n_seqs, n_heads, n_heads_kv, n_q, n_kv,
                                   head_dim_k, head_dim_v, scale};
    cudaError_t e;
    if (dtype == GDN_DTYPE_BF16)
        e = gdn::attn::launch_dtype<__nv_bfloat16>(p, st);
    else if (dtype == GDN_DTYPE_F16)
        e = gdn::attn::launch_dtype<__half>(p, st);
    else
        e = gdn::attn::launch_dtype<float>(p, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // extern "C"
