// Recurrent (token-by-token) path of the gated delta rule: the decode kernel.
//
// For one (sequence, head) the value rows of the state are independent of
// each other: row i of S (the keys seen from value component i) evolves as
//     s_k   = S[i,:] . k          s_q = S[i,:] . q          kq = k . q
//     alpha = exp(g)
//     delta = beta * (v_i - alpha * s_k)
//     S[i,:] <- alpha * S[i,:] + delta * k
//     o_i    = (alpha * s_q + delta * kq) / sqrt(d)
// which is S_t = alpha S_{t-1}(I - beta k k^T) + beta v k^T, o = S_t q / sqrt(d)
// restricted to one row: both dot products use the row before the update, so
// a single fused reduction per token serves the read (S k), the output (S q)
// and k.q.  ("marcsun13/ggml-gated-delta-net" model card, section "Ops":
// state [value][key] keeps a row contiguous, the output carries
// 1/sqrt(head_dim), g is exponentiated by the kernel.)
//
// Mapping on sm_103a: L lanes hold one state row in registers, each lane
// NV 128-bit vectors (4 fp32 keys) interleaved so that every load
// instruction of a warp covers whole 128-byte lines; a warp holds
// R * (32 / L) rows; a 128-thread block holds 4 warps' rows of one head.
// The row is loaded once, kept in registers for the whole token run, and
// written once: the state streams through HBM exactly once per call.  q, k,
// v, g, beta of the next token are prefetched while the current one is
// computed.
//
// Optional fused preprocessing (NORM): q and k are divided by their Euclidean
// norm per token before the recurrence.  The two squared norms join the same
// butterfly as the dot products, and the division is applied as scalars:
// S k^ = (S k) / |k|, S q^ = (S q) / |q|, k^.q^ = (k.q) / (|k| |q|), and the
// update adds (delta / |k|) k.  A zero vector stays zero (its scale is 0).
#include <cuda_bf16.h>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace gdn {
namespace {

// Raw 4-element vectors as loaded from memory.
struct Raw4F32 { float4 x; };
struct Raw4BF16 { uint2 x; };

template <typename Tin> struct RawOf;
template <> struct RawOf<float> { using type = Raw4F32; };
template <> struct RawOf<__nv_bfloat16> { using type = Raw4BF16; };

__device__ __forceinline__ Raw4F32 load_raw4(const float *p) {
    return {__ldg(reinterpret_cast<const float4 *>(p))};
}
__device__ __forceinline__ Raw4BF16 load_raw4(const __nv_bfloat16 *p) {
    return {__ldg(reinterpret_cast<const uint2 *>(p))};
}
__device__ __forceinline__ void unpack4(const Raw4F32 &r, float (&x)[4]) {
    x[0] = r.x.x; x[1] = r.x.y; x[2] = r.x.z; x[3] = r.x.w;
}
// bf16 -> fp32 is exact: the bf16 word is the upper half of the fp32 word.
__device__ __forceinline__ void unpack4(const Raw4BF16 &r, float (&x)[4]) {
    x[0] = __uint_as_float(r.x.x << 16);
    x[1] = __uint_as_float(r.x.x & 0xffff0000u);
    x[2] = __uint_as_float(r.x.y << 16);
    x[3] = __uint_as_float(r.x.y & 0xffff0000u);
}
__device__ __forceinline__ float load_scalar(const float *p) { return __ldg(p); }
__device__ __forceinline__ float load_scalar(const __nv_bfloat16 *p) {
    return __bfloat162float(__ldg(p));
}

// Warm L2 with `bytes` (a multiple of 16, 16-byte aligned) at `p`.  Only a
// hint: nothing is read into the program, so it may be issued before the
// previous grid has finished; L2 is the point of coherence, so lines that
// grid still writes are simply updated there.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Packed fp32 arithmetic on element pairs (sm_100 family): each element is
// rounded exactly as the scalar fmaf / multiplication rounds it.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

template <int D, int L, int R, typename Tin>
struct TokenInputs {
    static constexpr int NV = D / (4 * L);
    typename RawOf<Tin>::type q[NV], k[NV];
    float v[R];
    float g, beta;
};

// One output value: float32 as computed, or bf16 rounded to nearest even.
__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// 1 / |x| from the squared norm, 0 for a zero vector.
__device__ __forceinline__ float inv_norm(float sq) { return sq > 0.f ? rsqrtf(sq) : 0.f; }

template <int D, int L, int R, typename Tin, bool NORM, typename Tout>
__global__ void __launch_bounds__(128)
recurrent_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                 const Tin *__restrict__ v, const float *__restrict__ g,
                 const float *__restrict__ beta, const float *state_in,
                 float *state_out, Tout *__restrict__ out, int T, int H, int Hk,
                 float scale)
{
    constexpr int NV = D / (4 * L);   // 128-bit vectors per lane per row
    constexpr int RU = 32 / L;        // rows per warp unit
    constexpr int RW = R * RU;        // rows per warp
    constexpr int RB = 4 * RW;        // rows per block
    static_assert(D % RB == 0, "rows per block must divide head_dim");
    static_assert(NV >= 1 && D == NV * 4 * L, "bad lane split");

    // Launched with programmatic stream serialization: this grid may be
    // scheduled while the previous kernel on the stream is still running.
    // Nothing is read before the previous grid has completed and flushed; the
    // block's state rows (one contiguous run of RB rows) are only prefetched
    // into L2 meanwhile, so their HBM latency overlaps the previous kernel.
    if (threadIdx.x == 0 && state_in)
        prefetch_l2(state_in + (size_t)blockIdx.x * D * D + (size_t)blockIdx.y * RB * D,
                    RB * D * (uint32_t)sizeof(float));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int bh = blockIdx.x;  // b * H + h
    const int b = bh / H;
    const int h = bh - b * H;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int sub = lane % L;
    const int grp = lane / L;
    const int row0 = blockIdx.y * RB + warp * RW + grp;  // unit u owns row0 + u*RU

    // ---- state rows into registers --------------------------------------
    float s[R][NV][4];
    const size_t st_base = (size_t)bh * D * D;
#pragma unroll
    for (int u = 0; u < R; ++u) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if (state_in) {
                const float4 t = __ldcs(reinterpret_cast<const float4 *>(
                    state_in + st_base + (size_t)(row0 + u * RU) * D + (j * L + sub) * 4));
                s[u][j][0] = t.x; s[u][j][1] = t.y; s[u][j][2] = t.z; s[u][j][3] = t.w;
            } else {
                s[u][j][0] = s[u][j][1] = s[u][j][2] = s[u][j][3] = 0.f;
            }
        }
    }

    // value head h reads query / key head h % Hk (Hk == H: the identity)
    const size_t tok_stride = (size_t)H * D;                 // between tokens of one value head
    const size_t qk_stride = (size_t)Hk * D;                 // between tokens of one key head
    const size_t in_base = ((size_t)b * T * H + h) * D;      // token 0 of (b, h)
    const size_t qk_base = ((size_t)b * T * Hk + h % Hk) * D;
    const size_t gb_base = (size_t)b * T * H + h;
    const Tin *qp = q + qk_base;
    const Tin *kp = k + qk_base;
    const Tin *vp = v + in_base;
    const float *gp = g + gb_base;
    const float *bp = beta + gb_base;
    Tout *op = out + in_base;

    using In = TokenInputs<D, L, R, Tin>;
    auto load_token = [&](int t, In &x) {
        const size_t o = (size_t)t * tok_stride, oq = (size_t)t * qk_stride;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            x.q[j] = load_raw4(qp + oq + (j * L + sub) * 4);
            x.k[j] = load_raw4(kp + oq + (j * L + sub) * 4);
        }
#pragma unroll
        for (int u = 0; u < R; ++u) x.v[u] = load_scalar(vp + o + row0 + u * RU);
        x.g = __ldg(gp + (size_t)t * H);
        x.beta = __ldg(bp + (size_t)t * H);
    };

    In cur;
    load_token(0, cur);
    for (int t = 0; t < T; ++t) {
        In nxt;
        if (t + 1 < T) load_token(t + 1, nxt);

        float qv[NV][4], kv[NV][4];
#pragma unroll
        for (int j = 0; j < NV; ++j) { unpack4(cur.q[j], qv[j]); unpack4(cur.k[j], kv[j]); }

        float kq = 0.f, pk[R], pq[R], qq = 0.f, kk = 0.f;
#pragma unroll
        for (int u = 0; u < R; ++u) { pk[u] = 0.f; pq[u] = 0.f; }
#pragma unroll
        for (int j = 0; j < NV; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kq = fmaf(kv[j][e], qv[j][e], kq);
                if constexpr (NORM) {
                    qq = fmaf(qv[j][e], qv[j][e], qq);
                    kk = fmaf(kv[j][e], kv[j][e], kk);
                }
#pragma unroll
                for (int u = 0; u < R; ++u) {
                    pk[u] = fmaf(s[u][j][e], kv[j][e], pk[u]);
                    pq[u] = fmaf(s[u][j][e], qv[j][e], pq[u]);
                }
            }
        }
        // butterfly over the L lanes of each row group: every lane gets the sums
#pragma unroll
        for (int off = L / 2; off > 0; off >>= 1) {
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
            if constexpr (NORM) {
                qq += __shfl_xor_sync(0xffffffffu, qq, off);
                kk += __shfl_xor_sync(0xffffffffu, kk, off);
            }
#pragma unroll
            for (int u = 0; u < R; ++u) {
                pk[u] += __shfl_xor_sync(0xffffffffu, pk[u], off);
                pq[u] += __shfl_xor_sync(0xffffffffu, pq[u], off);
            }
        }
        float ik = 1.f;                               // 1 / |k| (NORM), else 1
        if constexpr (NORM) {
            ik = inv_norm(kk);
            const float iq = inv_norm(qq);
            kq *= ik * iq;
#pragma unroll
            for (int u = 0; u < R; ++u) { pk[u] *= ik; pq[u] *= iq; }
        }

        const float alpha = expf(cur.g);
        const size_t o = (size_t)t * tok_stride;
#pragma unroll
        for (int u = 0; u < R; ++u) {
            const float delta = cur.beta * (cur.v[u] - alpha * pk[u]);
            const float dk = NORM ? delta * ik : delta;   // the update adds delta k^
#pragma unroll
            for (int j = 0; j < NV; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    s[u][j][e] = fmaf(alpha, s[u][j][e], dk * kv[j][e]);
            const float ov = fmaf(alpha, pq[u], delta * kq) * scale;
            if (sub == 0) store_out(op + o + row0 + u * RU, ov);
        }
        if (t + 1 < T) cur = nxt;
    }

    // ---- state rows back --------------------------------------------------
#pragma unroll
    for (int u = 0; u < R; ++u)
#pragma unroll
        for (int j = 0; j < NV; ++j)
            __stcs(reinterpret_cast<float4 *>(state_out + st_base + (size_t)(row0 + u * RU) * D +
                                              (j * L + sub) * 4),
                   make_float4(s[u][j][0], s[u][j][1], s[u][j][2], s[u][j][3]));
}

// ---------------------------------------------------------------------------
// Multi-token runs (T >= 2).  The per-token work is short (three dot
// products over a row, a butterfly, one update), so with a one-token
// prefetch the loop waits on global-memory latency at every token.  Here the
// inputs of WT consecutive tokens (q, k of the key head, the block's slice of
// v, g, beta) are staged in shared memory by asynchronous copies, two windows
// in flight: window w + 1 streams in while window w is computed.  The state
// rows stay in registers for the whole run, exactly as in recurrent_kernel.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_prev() {   // all but the latest group landed
    asm volatile("cp.async.wait_group 1;" ::: "memory");
}

__device__ __forceinline__ Raw4F32 lds_raw4(const float *p) {
    return {*reinterpret_cast<const float4 *>(p)};
}
__device__ __forceinline__ Raw4BF16 lds_raw4(const __nv_bfloat16 *p) {
    return {*reinterpret_cast<const uint2 *>(p)};
}
__device__ __forceinline__ float lds_scalar(const float *p) { return *p; }
__device__ __forceinline__ float lds_scalar(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <int D, int RB, typename Tin, int WT>
struct alignas(16) TokenWindow {
    Tin q[WT][D];
    Tin k[WT][D];
    Tin v[WT][RB];
    float g[WT];
    float beta[WT];
    float kq[WT];      // k . q of each token (of the normalised q, k with NORM)
    float alpha[WT];   // exp(g) of each token
    float ik[WT];      // 1 / |k| of each token (NORM)
    float iq[WT];      // 1 / |q| of each token (NORM)
};

template <int D, int L, int R, typename Tin, int WT, bool NORM, typename Tout>
__global__ void __launch_bounds__(128)
recurrent_window_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                        const Tin *__restrict__ v, const float *__restrict__ g,
                        const float *__restrict__ beta, const float *state_in,
                        float *state_out, Tout *__restrict__ out, int T, int H, int Hk,
                        float scale)
{
    constexpr int NV = D / (4 * L);
    constexpr int RU = 32 / L;
    constexpr int RW = R * RU;
    constexpr int RB = 4 * RW;
    constexpr int EPC = 16 / (int)sizeof(Tin);              // elements per 16-byte copy
    constexpr int CPR = D / EPC;                            // copies per q (or k) row
    constexpr int CPV = RB / EPC;                           // copies per token's v slice
    static_assert(D % RB == 0 && NV >= 1 && D == NV * 4 * L, "bad lane split");
    static_assert(RB % EPC == 0, "v slice must be whole 16-byte copies");
    static_assert(WT <= 64, "g / beta copies use threads 0..WT-1 and 64..64+WT-1");
    using Win = TokenWindow<D, RB, Tin, WT>;
    __shared__ Win win[2];

    if (threadIdx.x == 0 && state_in)                       // as in recurrent_kernel
        prefetch_l2(state_in + (size_t)blockIdx.x * D * D + (size_t)blockIdx.y * RB * D,
                    RB * D * (uint32_t)sizeof(float));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int bh = blockIdx.x;
    const int b = bh / H;
    const int h = bh - b * H;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int sub = lane % L;
    const int grp = lane / L;
    const int lrow0 = warp * RW + grp;                      // row within the block
    const int row0 = blockIdx.y * RB + lrow0;

    float s[R][NV][4];
    const size_t st_base = (size_t)bh * D * D;
#pragma unroll
    for (int u = 0; u < R; ++u) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            if (state_in) {
                const float4 t = __ldcs(reinterpret_cast<const float4 *>(
                    state_in + st_base + (size_t)(row0 + u * RU) * D + (j * L + sub) * 4));
                s[u][j][0] = t.x; s[u][j][1] = t.y; s[u][j][2] = t.z; s[u][j][3] = t.w;
            } else {
                s[u][j][0] = s[u][j][1] = s[u][j][2] = s[u][j][3] = 0.f;
            }
        }
    }

    const size_t tok_stride = (size_t)H * D;
    const size_t qk_stride = (size_t)Hk * D;
    const Tin *qp = q + ((size_t)b * T * Hk + h % Hk) * D;
    const Tin *kp = k + ((size_t)b * T * Hk + h % Hk) * D;
    const Tin *vp = v + ((size_t)b * T * H + h) * D + blockIdx.y * RB;
    const float *gp = g + (size_t)b * T * H + h;
    const float *bp = beta + (size_t)b * T * H + h;
    Tout *op = out + ((size_t)b * T * H + h) * D;

    // stage window w (tokens w*WT .. min(T, (w+1)*WT) - 1) into buffer `buf`
    auto issue = [&](int w, int buf) {
        const int t0 = w * WT;
        const int nt = min(WT, T - t0);
        Win &W_ = win[buf];
        for (int i = tid; i < 2 * WT * CPR; i += 128) {
            const int which = i / (WT * CPR), rem = i - which * (WT * CPR);
            const int j = rem / CPR, c = rem - j * CPR;
            if (j < nt) {
                const Tin *src = (which ? kp : qp) + (size_t)(t0 + j) * qk_stride + c * EPC;
                cp_async16(which ? &W_.k[j][c * EPC] : &W_.q[j][c * EPC], src);
            }
        }
        for (int i = tid; i < WT * CPV; i += 128) {
            const int j = i / CPV, c = i - j * CPV;
            if (j < nt) cp_async16(&W_.v[j][c * EPC], vp + (size_t)(t0 + j) * tok_stride + c * EPC);
        }
        if (tid < nt) cp_async4(&W_.g[tid], gp + (size_t)(t0 + tid) * H);
        else if (tid >= 64 && tid - 64 < nt) cp_async4(&W_.beta[tid - 64], bp + (size_t)(t0 + tid - 64) * H);
        cp_async_commit();
    };

    const int n_win = (T + WT - 1) / WT;
    issue(0, 0);
    for (int w = 0; w < n_win; ++w) {
        if (w + 1 < n_win) issue(w + 1, (w + 1) & 1);
        else cp_async_commit();                              // keep the group count uniform
        cp_async_wait_prev();
        __syncthreads();                                     // window w visible to all
        Win &W_ = win[w & 1];
        const int t0 = w * WT;
        const int nt = min(WT, T - t0);
        // the per-token scalars every row needs, once per token: one warp each
        for (int j = warp; j < nt; j += 4) {
            float acc = 0.f, qq = 0.f, kk = 0.f;
#pragma unroll
            for (int e = lane; e < D; e += 32) {
                const float qe = lds_scalar(&W_.q[j][e]), ke = lds_scalar(&W_.k[j][e]);
                acc = fmaf(qe, ke, acc);
                if constexpr (NORM) {
                    qq = fmaf(qe, qe, qq);
                    kk = fmaf(ke, ke, kk);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if constexpr (NORM) {
                    qq += __shfl_xor_sync(0xffffffffu, qq, off);
                    kk += __shfl_xor_sync(0xffffffffu, kk, off);
                }
            }
            if (lane == 0) {
                if constexpr (NORM) {
                    const float ik = inv_norm(kk), iq = inv_norm(qq);
                    W_.ik[j] = ik;
                    W_.iq[j] = iq;
                    acc *= ik * iq;
                }
                W_.kq[j] = acc;
                W_.alpha[j] = expf(W_.g[j]);
            }
        }
        __syncthreads();
        for (int j = 0; j < nt; ++j) {
            float qv[NV][4], kv[NV][4];
#pragma unroll
            for (int jv = 0; jv < NV; ++jv) {
                unpack4(lds_raw4(&W_.q[j][(jv * L + sub) * 4]), qv[jv]);
                unpack4(lds_raw4(&W_.k[j][(jv * L + sub) * 4]), kv[jv]);
            }
            // S k and S q on this lane's slice, element pairs in packed FMAs
            float pk[R], pq[R];
#pragma unroll
            for (int u = 0; u < R; ++u) {
                float2 ak = make_float2(0.f, 0.f), aq = make_float2(0.f, 0.f);
#pragma unroll
                for (int jv = 0; jv < NV; ++jv) {
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const float2 sv = make_float2(s[u][jv][e], s[u][jv][e + 1]);
                        ak = ffma2(sv, make_float2(kv[jv][e], kv[jv][e + 1]), ak);
                        aq = ffma2(sv, make_float2(qv[jv][e], qv[jv][e + 1]), aq);
                    }
                }
                pk[u] = ak.x + ak.y;
                pq[u] = aq.x + aq.y;
            }
#pragma unroll
            for (int off = L / 2; off > 0; off >>= 1) {
#pragma unroll
                for (int u = 0; u < R; ++u) {
                    pk[u] += __shfl_xor_sync(0xffffffffu, pk[u], off);
                    pq[u] += __shfl_xor_sync(0xffffffffu, pq[u], off);
                }
            }
            const float alpha = W_.alpha[j];
            const float kq = W_.kq[j];
            const float bt = W_.beta[j];
            const size_t o = (size_t)(t0 + j) * tok_stride;
            float ik = 1.f;
            if constexpr (NORM) {
                ik = W_.ik[j];
                const float iq = W_.iq[j];
#pragma unroll
                for (int u = 0; u < R; ++u) { pk[u] *= ik; pq[u] *= iq; }
            }
#pragma unroll
            for (int u = 0; u < R; ++u) {
                const float vv = lds_scalar(&W_.v[j][lrow0 + u * RU]);
                const float delta = bt * (vv - alpha * pk[u]);
                const float dk = NORM ? delta * ik : delta;    // the update adds delta k^
                const float2 a2 = make_float2(alpha, alpha), d2 = make_float2(dk, dk);
#pragma unroll
                for (int jv = 0; jv < NV; ++jv)
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        // s <- alpha s + delta k, as the scalar fmaf(alpha, s, delta * k)
                        const float2 dk = fmul2(d2, make_float2(kv[jv][e], kv[jv][e + 1]));
                        const float2 sn = ffma2(a2, make_float2(s[u][jv][e], s[u][jv][e + 1]), dk);
                        s[u][jv][e] = sn.x;
                        s[u][jv][e + 1] = sn.y;
                    }
                const float ov = fmaf(alpha, pq[u], delta * kq) * scale;
                if (sub == 0) store_out(op + o + row0 + u * RU, ov);
            }
        }
        __syncthreads();                                     // buffer w & 1 free for window w + 2
    }

#pragma unroll
    for (int u = 0; u < R; ++u)
#pragma unroll
        for (int j = 0; j < NV; ++j)
            __stcs(reinterpret_cast<float4 *>(state_out + st_base + (size_t)(row0 + u * RU) * D +
                                              (j * L + sub) * 4),
                   make_float4(s[u][j][0], s[u][j][1], s[u][j][2], s[u][j][3]));
}

// Tokens staged per window by the multi-token kernel.
constexpr int kWindow = 8;

template <int D, int L, int R, typename Tin, bool NORM, typename Tout>
cudaError_t launch_one_out(const Problem &p, cudaStream_t stream) {
    constexpr int RB = 4 * R * (32 / L);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.B * (unsigned)p.H, D / RB);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    // back-to-back calls (e.g. the layers of one decode step) overlap launch
    // latency with the tail of the previous kernel
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.T >= 2)
        return cudaLaunchKernelEx(&cfg, recurrent_window_kernel<D, L, R, Tin, kWindow, NORM, Tout>,
                                  static_cast<const Tin *>(p.q), static_cast<const Tin *>(p.k),
                                  static_cast<const Tin *>(p.v), p.g, p.beta, p.state_in,
                                  p.state_out, reinterpret_cast<Tout *>(p.out), p.T, p.H, p.Hk,
                                  p.scale);
    return cudaLaunchKernelEx(&cfg, recurrent_kernel<D, L, R, Tin, NORM, Tout>,
                              static_cast<const Tin *>(p.q), static_cast<const Tin *>(p.k),
                              static_cast<const Tin *>(p.v), p.g, p.beta, p.state_in, p.state_out,
                              reinterpret_cast<Tout *>(p.out), p.T, p.H, p.Hk, p.scale);
}

// The output type is a template parameter: with a runtime switch the
// multi-token kernel needed 9 more registers and lost one block per SM.
template <int D, int L, int R, typename Tin, bool NORM>
cudaError_t launch_one(const Problem &p, cudaStream_t stream) {
    return p.out_bf16 ? launch_one_out<D, L, R, Tin, NORM, __nv_bfloat16>(p, stream)
                      : launch_one_out<D, L, R, Tin, NORM, float>(p, stream);
}

template <int D, int L, typename Tin, bool NORM>
cudaError_t launch_d(const Problem &p, cudaStream_t stream) {
    // Two rows per warp unit when there are enough blocks to fill the GPU
    // several times over (more bytes in flight per thread); one otherwise.
    constexpr int RB2 = 4 * 2 * (32 / L);
    const long long blocks2 = (long long)p.B * p.H * (D / RB2);
    if (D % RB2 == 0 && blocks2 >= 4LL * current_sm_count())
        return launch_one<D, L, 2, Tin, NORM>(p, stream);
    return launch_one<D, L, 1, Tin, NORM>(p, stream);
}

template <typename Tin, bool NORM>
cudaError_t launch_dtype(const Problem &p, cudaStream_t stream) {
    switch (p.d) {
        case 32: return launch_one<32, 8, 1, Tin, NORM>(p, stream);
        case 64: return launch_d<64, 8, Tin, NORM>(p, stream);
        case 96: return launch_d<96, 8, Tin, NORM>(p, stream);
        case 128: return launch_d<128, 8, Tin, NORM>(p, stream);
        case 256: return launch_d<256, 16, Tin, NORM>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_recurrent(const Problem &p, cudaStream_t stream) {
    if (p.dtype == GDN_DTYPE_BF16)
        return p.l2norm_qk ? launch_dtype<__nv_bfloat16, true>(p, stream)
                           : launch_dtype<__nv_bfloat16, false>(p, stream);
    return p.l2norm_qk ? launch_dtype<float, true>(p, stream) : launch_dtype<float, false>(p, stream);
}

}  // namespace gdn
