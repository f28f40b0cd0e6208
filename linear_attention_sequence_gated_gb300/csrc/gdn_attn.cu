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
// the kernel is bound by HBM and by latency, not by arithmetic.  Mapping on
// sm_103a:
//   * the R = (n_heads / n_heads_kv) * n_q rows of one kv head are cut into
//     row groups of RG rows; one thread-block cluster of CL <= 8 CTAs serves
//     (sequence, kv head, row block), and the cluster's CL x (warps per row
//     group) warps split the keys into contiguous ranges;
//   * a warp streams its keys eight at a time through its own ring of
//     shared-memory stages filled by asynchronous copies (two steps of k and v
//     in flight while one is computed, no block barrier), lanes splitting
//     head_dim, and keeps its own online softmax (running max, sum of exp,
//     output slice) per row;
//   * the eight keys' partial dot products are reduced across the warp by a
//     transposing butterfly (about one shuffle per key and row);
//   * at the end the warps of a CTA merge through shared memory and the CTAs
//     of the cluster through distributed shared memory, so no partial result
//     goes through global scratch.
// Accumulation is fp32 from exactly upcast inputs (upstream accumulates in
// f16; that is its kernel's choice, not part of the operation).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace attn {
namespace {

constexpr int KG = 8;           // keys per step of a warp
constexpr int MAX_CLUSTER = 8;  // portable cluster size

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

// A lane's SL consecutive elements of one row (SL = head_dim / 32), raw.
template <typename Tin, int SL>
struct Slice {
    static constexpr int BYTES = SL * (int)sizeof(Tin);
    static constexpr int WORDS = BYTES / 4;
    uint32_t w[WORDS];
};
// from global memory (kGlobal) or shared memory
template <bool kGlobal, typename Tin, int SL>
__device__ __forceinline__ void ld_slice(Slice<Tin, SL> &s, const Tin *p) {
    constexpr int B = Slice<Tin, SL>::BYTES;
    if constexpr (B == 4) {
        s.w[0] = kGlobal ? __ldg(reinterpret_cast<const uint32_t *>(p))
                         : *reinterpret_cast<const uint32_t *>(p);
    } else if constexpr (B == 8) {
        const uint2 a = kGlobal ? __ldg(reinterpret_cast<const uint2 *>(p))
                                : *reinterpret_cast<const uint2 *>(p);
        s.w[0] = a.x; s.w[1] = a.y;
    } else {
#pragma unroll
        for (int i = 0; i < B / 16; ++i) {
            const uint4 a = kGlobal ? __ldg(reinterpret_cast<const uint4 *>(p) + i)
                                    : *(reinterpret_cast<const uint4 *>(p) + i);
            s.w[4 * i] = a.x; s.w[4 * i + 1] = a.y; s.w[4 * i + 2] = a.z; s.w[4 * i + 3] = a.w;
        }
    }
}
template <int SL>
__device__ __forceinline__ void unpack(const Slice<float, SL> &s, float (&x)[SL]) {
#pragma unroll
    for (int i = 0; i < SL; ++i) x[i] = __uint_as_float(s.w[i]);
}
template <int SL>
__device__ __forceinline__ void unpack(const Slice<__nv_bfloat16, SL> &s, float (&x)[SL]) {
#pragma unroll
    for (int i = 0; i < SL / 2; ++i) {
        x[2 * i] = __uint_as_float(s.w[i] << 16);
        x[2 * i + 1] = __uint_as_float(s.w[i] & 0xffff0000u);
    }
}
template <int SL>
__device__ __forceinline__ void unpack(const Slice<__half, SL> &s, float (&x)[SL]) {
#pragma unroll
    for (int i = 0; i < SL / 2; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&s.w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

// Geometry for head_dim D and input type Tin.  A warp keeps RG rows' query
// slice, output slice and one step's partial dot products in registers; its
// ring holds ST steps of KG keys of k and v.  Eight warps and three stages
// unless that ring would not fit, then four warps and two stages.
template <int D, typename Tin> struct Geo {
    static constexpr int ELT = (int)sizeof(Tin);
    static constexpr int SL = D / 32;                 // elements of a row per lane
    static constexpr int RG = D == 256 ? 2 : 4;       // rows per warp
    static constexpr int STEP = KG * 2 * D * ELT;     // bytes of one step: k rows, then v rows
    static constexpr bool BIG = 8 * 3 * STEP > 200 * 1024;
    static constexpr int NW = BIG ? 4 : 8;            // warps per CTA
    static constexpr int ST = BIG ? 2 : 3;            // ring stages per warp
    static constexpr int NTHR = NW * 32;
    static constexpr int RING = NW * ST * STEP;
    // after the key loop the ring is reused for the merge buffers
    static constexpr int WO = 0;                                  // [NW][RG][D] fp32
    static constexpr int CO = WO + NW * RG * D * 4;               // [NW*RG][D] fp32
    static constexpr int SMEM = RING > CO + NW * RG * D * 4 ? RING : CO + NW * RG * D * 4;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static constexpr int MIN_CTAS = SMEM <= 110 * 1024 ? 2 : 1;   // CTAs an SM should hold
};

// Small per-CTA state outside the ring.
template <int NW, int RG>
struct SmallSmem {
    float wm[NW][RG], wl[NW][RG];                     // each warp's partial max, sum per row
    float cm[NW * RG], cl[NW * RG];                   // the CTA's partial per local row
    float p[NW][RG][KG];                              // a step's probabilities, per warp
};

template <int D, typename Tin>
__global__ void __launch_bounds__(Geo<D, Tin>::NTHR, Geo<D, Tin>::MIN_CTAS)
attn_decode_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                   const Tin *__restrict__ v, const Tin *__restrict__ mask,
                   float *__restrict__ out, int H, int Hkv, int n_q, int n_kv, int n_rb, int n_rgc,
                   int CL, float scale)
{
    using G = Geo<D, Tin>;
    constexpr int SL = G::SL, RG = G::RG, NW = G::NW, ST = G::ST, NTHR = G::NTHR;
    constexpr int NWARP = NW;
    extern __shared__ __align__(16) uint8_t ring[];
    __shared__ SmallSmem<NW, RG> sm;
    float (*wo)[RG][D] = reinterpret_cast<float (*)[RG][D]>(ring + G::WO);
    float (*co)[D] = reinterpret_cast<float (*)[D]>(ring + G::CO);

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
    const int n_ksc = NWARP / n_rgc;                  // warps per row group in a CTA
    const int rgc = warp % n_rgc;                     // this warp's row group in the CTA
    const int ksw = warp / n_rgc;                     // this warp's key split in the CTA
    const int rows_cta = n_rgc * RG;
    const int r0 = rb * rows_cta + rgc * RG;          // first row of this warp
    const int nr = max(0, min(RG, R - r0));

    // key range of this warp: split s of S = CL * n_ksc, in steps of KG
    const int S = CL * n_ksc;
    const int s = rank * n_ksc + ksw;
    const int n_steps_all = (n_kv + KG - 1) / KG;
    const int sps = (n_steps_all + S - 1) / S;
    const int kb = min(n_kv, s * sps * KG);
    const int ke = min(n_kv, kb + sps * KG);

    // this lane's slice of the warp's rows of q, scaled, fp32
    float qv[RG][SL];
#pragma unroll
    for (int r = 0; r < RG; ++r) {
        if (r < nr) {
            const int rg = r0 + r;                    // head hk*rep + rg / n_q, query rg % n_q
            Slice<Tin, SL> raw;
            ld_slice<true>(raw, q + ((size_t)(b * H + hk * rep) * n_q + rg) * D + lane * SL);
            unpack(raw, qv[r]);
#pragma unroll
            for (int e = 0; e < SL; ++e) qv[r][e] *= scale;
        } else {
#pragma unroll
            for (int e = 0; e < SL; ++e) qv[r][e] = 0.f;
        }
    }
    float m[RG], l[RG], acc[RG][SL];
#pragma unroll
    for (int r = 0; r < RG; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < SL; ++e) acc[r][e] = 0.f;
    }

    const Tin *kg = k + (size_t)(b * Hkv + hk) * n_kv * D;
    const Tin *vg = v + (size_t)(b * Hkv + hk) * n_kv * D;
    uint8_t *wring = ring + warp * ST * G::STEP;
    const int n_steps = nr > 0 ? (ke - kb + KG - 1) / KG : 0;
    // stage `st` <- keys kb + KG*step .. (k rows, then v rows); rows past the
    // range are not copied (their scores are masked, their v rows skipped)
    auto issue = [&](int step, int st) {
        if (step < n_steps) {
            const int j0 = kb + step * KG;
            const int nk = min(KG, ke - j0);
            constexpr int CPR = D * G::ELT / 16;      // 16-byte copies per row
            uint8_t *dst = wring + st * G::STEP;
            for (int c = lane; c < KG * CPR; c += 32) {
                const int g = c / CPR, x = c - g * CPR;
                if (g < nk) {
                    cp_async16(dst + g * D * G::ELT + x * 16,
                               reinterpret_cast<const uint8_t *>(kg + (size_t)(j0 + g) * D) + x * 16);
                    cp_async16(dst + (KG + g) * D * G::ELT + x * 16,
                               reinterpret_cast<const uint8_t *>(vg + (size_t)(j0 + g) * D) + x * 16);
                }
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < ST - 1; ++i) issue(i, i);

    for (int step = 0; step < n_steps; ++step) {
        cp_async_wait<ST - 2>();                      // this step's copies (own lane) landed
        __syncwarp();                                 // ... and every lane's
        const int j0 = kb + step * KG;
        const int nk = min(KG, ke - j0);
        const Tin *sk = reinterpret_cast<const Tin *>(wring + (step % ST) * G::STEP);
        const Tin *sv = sk + KG * D;
        Slice<Tin, SL> kr[KG];
#pragma unroll
        for (int g = 0; g < KG; ++g) ld_slice<false>(kr[g], sk + g * D + lane * SL);
        // partial dot products of this lane's slice: part[r][g]
        float part[RG][KG];
#pragma unroll
        for (int g = 0; g < KG; ++g) {
            float kx[SL];
            unpack(kr[g], kx);
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < SL; ++e) a = fmaf(qv[r][e], kx[e], a);
                part[r][g] = a;
            }
        }
        // transposing butterfly: after the xor-16/8/4 steps lane holds the sum
        // over its 8-lane class for key kidx; xor-2/1 finish the sum over all 32
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
            float h4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                // keys i (bit 2 of key = 0 half) vs i + 4: keep own half
                const float keep = b4 ? part[r][i + 4] : part[r][i];
                const float send = b4 ? part[r][i] : part[r][i + 4];
                h4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
            float h2[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float keep = b3 ? h4[i + 2] : h4[i];
                const float send = b3 ? h4[i] : h4[i + 2];
                h2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
            float h1;
            {
                const float keep = b2 ? h2[1] : h2[0];
                const float send = b2 ? h2[0] : h2[1];
                h1 = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
            h1 += __shfl_xor_sync(0xffffffffu, h1, 2);
            h1 += __shfl_xor_sync(0xffffffffu, h1, 1);
            // h1 is the score of key (b4 ? 4 : 0) + (b3 ? 2 : 0) + (b2 ? 1 : 0)
            const int key = (b4 ? 4 : 0) + (b3 ? 2 : 0) + (b2 ? 1 : 0);
            float sc = h1;
            if (key < nk) {
                if (mask) {
                    const int i = (r0 + r) % n_q;
                    sc += to_f32(mask[((size_t)b * n_q + i) * n_kv + j0 + key]);
                }
            } else {
                sc = -INFINITY;
            }
            float gm = sc;
            gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 4));
            gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 8));
            gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, 16));
            const float m_new = fmaxf(m[r], gm);
            const bool none = (m_new == -INFINITY);
            const float p = none ? 0.f : expf(sc - m_new);
            float ps = p;
            ps += __shfl_xor_sync(0xffffffffu, ps, 4);
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            const float c = none ? 1.f : expf(m[r] - m_new);
            m[r] = m_new;
            l[r] = fmaf(l[r], c, ps);
#pragma unroll
            for (int e = 0; e < SL; ++e) acc[r][e] *= c;
            if ((lane & 3) == 0) sm.p[warp][r][key] = p;
        }
        __syncwarp();
        // P V on this lane's slice (keys past the range are skipped: their
        // stage rows hold stale data)
#pragma unroll
        for (int g = 0; g < KG; ++g) {
            if (g < nk) {
                Slice<Tin, SL> vr;
                ld_slice<false>(vr, sv + g * D + lane * SL);
                float vx[SL];
                unpack(vr, vx);
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    const float p = sm.p[warp][r][g];
#pragma unroll
                    for (int e = 0; e < SL; ++e) acc[r][e] = fmaf(p, vx[e], acc[r][e]);
                }
            }
        }
        __syncwarp();                                 // stage and probabilities consumed
        issue(step + ST - 1, (step + ST - 1) % ST);
    }
    cp_async_wait<0>();
    __syncthreads();                                  // every warp is done with the ring

    // ---- merge the warps of this CTA (same row group, different keys)
#pragma unroll
    for (int r = 0; r < RG; ++r) {
        if (lane == 0) { sm.wm[warp][r] = m[r]; sm.wl[warp][r] = l[r]; }
#pragma unroll
        for (int e = 0; e < SL; ++e) wo[warp][r][lane * SL + e] = acc[r][e];
    }
    __syncthreads();
    // CTA partial for local row lr = rgc * RG + r: merge warps ksw' * n_rgc + rgc
    for (int it = tid; it < rows_cta * D; it += NTHR) {
        const int lr = it / D, col = it - lr * D;
        const int g = lr / RG, r = lr - g * RG;
        float M = -INFINITY;
        for (int w = g; w < NWARP; w += n_rgc) M = fmaxf(M, sm.wm[w][r]);
        float L = 0.f, o = 0.f;
        if (M != -INFINITY) {
            for (int w = g; w < NWARP; w += n_rgc) {
                const float mw = sm.wm[w][r];
                if (mw != -INFINITY) {
                    const float wt = expf(mw - M);
                    L = fmaf(wt, sm.wl[w][r], L);
                    o = fmaf(wt, wo[w][r][col], o);
                }
            }
        }
        co[lr][col] = o;
        if (col == 0) { sm.cm[lr] = M; sm.cl[lr] = L; }
    }
    // ---- merge the CTAs of the cluster (same rows, different keys)
    cluster_sync();
    const int rbase = rb * rows_cta;
    const int nr_cta = max(0, min(rows_cta, R - rbase));
    for (int it = rank * NTHR + tid; it < nr_cta * D; it += CL * NTHR) {
        const int lr = it / D, col = it - lr * D;
        float mk[MAX_CLUSTER];
        float M = -INFINITY;
#pragma unroll
        for (int pr = 0; pr < MAX_CLUSTER; ++pr) {
            mk[pr] = pr < CL ? ld_peer(peer_addr(&sm.cm[lr], pr)) : -INFINITY;
            M = fmaxf(M, mk[pr]);
        }
        float L = 0.f, o = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int pr = 0; pr < MAX_CLUSTER; ++pr) {
                if (pr < CL && mk[pr] != -INFINITY) {
                    const float wt = expf(mk[pr] - M);
                    L = fmaf(wt, ld_peer(peer_addr(&sm.cl[lr], pr)), L);
                    o = fmaf(wt, ld_peer(peer_addr(&co[lr][col], pr)), o);
                }
            }
        }
        const int rg = rbase + lr;
        const int h = hk * rep + rg / n_q, i = rg % n_q;
        out[(((size_t)b * n_q + i) * H + h) * D + col] = (L > 0.f) ? o / L : 0.f;
    }
    cluster_sync();                                   // peers are done reading this CTA
}

struct AttnProblem {
    const void *q, *k, *v, *mask;
    float *out;
    int B, H, Hkv, n_q, n_kv, d;
    float scale;
};

template <int D, typename Tin>
cudaError_t launch(const AttnProblem &p, cudaStream_t stream) {
    using G = Geo<D, Tin>;
    constexpr int RG = G::RG, NWARP = G::NW;
    const int rep = p.H / p.Hkv;
    const long long R = (long long)rep * p.n_q;
    // row groups per CTA: enough for the rows, a power of two dividing 8
    int n_rgc = 1;
    while (n_rgc < NWARP && (long long)n_rgc * RG < R) n_rgc *= 2;
    const int n_ksc = NWARP / n_rgc;
    const int n_rb = (int)((R + (long long)n_rgc * RG - 1) / ((long long)n_rgc * RG));
    // CTAs per cluster: as many as give every warp at least one step of keys
    // (a short cache is latency-bound: spread it over as many SMs as allowed)
    const long long per_cta = (long long)n_ksc * KG;
    const long long want = (p.n_kv + per_cta - 1) / per_cta;
    const int CL = (int)(want < 1 ? 1 : (want > MAX_CLUSTER ? MAX_CLUSTER : want));
    const long long blocks = (long long)p.B * p.Hkv * n_rb * CL;
    if (blocks > INT_MAX) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_decode_kernel<D, Tin>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    });
    if (attr_err != cudaSuccess) return attr_err;
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
    return cudaLaunchKernelEx(&cfg, attn_decode_kernel<D, Tin>, static_cast<const Tin *>(p.q),
                              static_cast<const Tin *>(p.k), static_cast<const Tin *>(p.v),
                              static_cast<const Tin *>(p.mask), p.out, p.H, p.Hkv, p.n_q, p.n_kv,
                              n_rb, n_rgc, CL, p.scale);
}

template <typename Tin>
cudaError_t launch_dtype(const AttnProblem &p, cudaStream_t stream) {
    switch (p.d) {
        case 64: return launch<64, Tin>(p, stream);
        case 128: return launch<128, Tin>(p, stream);
        case 256: return launch<256, Tin>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

constexpr int kMaxQueries = 19;   // the vector (decode) variant: fewer than 20 queries

bool head_dims_ok(int dk, int dv) { return dk == dv && (dk == 64 || dk == 128 || dk == 256); }

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
    const unsigned long long d = (unsigned long long)head_dim_k;
    unsigned long long nq_rows, kv_rows, mask_n, q_bytes, kv_bytes, mask_bytes, out_bytes;
    if (!mul_ok((unsigned long long)n_seqs * (unsigned long long)n_heads, (unsigned long long)n_q,
                &nq_rows) ||
        !mul_ok((unsigned long long)n_seqs * (unsigned long long)n_heads_kv,
                (unsigned long long)n_kv, &kv_rows) ||
        !mul_ok((unsigned long long)n_seqs * (unsigned long long)n_q, (unsigned long long)n_kv,
                &mask_n))
        return GDN_ERR_ARG;
    unsigned long long nq_elems, kv_elems;
    if (!mul_ok(nq_rows, d, &nq_elems) || !mul_ok(kv_rows, d, &kv_elems) ||
        !span_bytes(nq_elems, elt, &q_bytes) || !span_bytes(kv_elems, elt, &kv_bytes) ||
        !span_bytes(mask_n, elt, &mask_bytes) || !span_bytes(nq_elems, 4, &out_bytes))
        return GDN_ERR_ARG;
    if (nq_rows == 0) return GDN_OK;                  // no queries: nothing to do
    if (!q || !out || (kv_rows > 0 && (!k || !v))) return GDN_ERR_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || (k && !aligned(k, 16)) || (v && !aligned(v, 16)) ||
        (mask && !aligned(mask, elt)))
        return GDN_ERR_ALIGN;
    const Range ro = range_of(out, out_bytes);
    for (Range in : {range_of(q, q_bytes), range_of(k, kv_bytes), range_of(v, kv_bytes),
                     range_of(mask, mask ? mask_bytes : 0)})
        if (overlap(ro, in)) return GDN_ERR_ALIAS;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (n_kv == 0)   // empty cache: every output row is zero
        return cudaMemsetAsync(out, 0, out_bytes, st) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    const gdn::attn::AttnProblem p{q, k, v, mask, out, n_seqs, n_heads, n_heads_kv, n_q, n_kv,
                                   head_dim_k, scale};
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
