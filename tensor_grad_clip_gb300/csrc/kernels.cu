// The kernels of one optimizer step (sm_103a).
//
//  norm_kernel   -- owned square-sum.  Every CTA walks chunks of the norm
//                   table, sums g^2 of its chunk in fp32 (per-thread
//                   accumulators, then a fixed-shape warp/block tree) and
//                   stores the chunk's sum at partials[chunk].  The last CTA
//                   to arrive (atomic ticket; nobody waits) adds the partials
//                   in fp64 in a fixed order, so the norm is the same bits
//                   on every run whatever the CTA schedule, then derives
//                   norm = sqrt(S) * (1/d) and c = min(1, max_norm/(norm + 1e-6)).
//                   It gathers what the SomaSpeed optimizer paragraphs need
//                   for one clipping decision over the whole list, with
//                   ownership resolved by the host (only owned segments are
//                   in this table).
//
//  update_kernel -- the fused normalize + clip + AdamW pass.  It reads the
//                   scale c/d that the norm kernel left in device memory (no
//                   host round trip) and streams every trainable element once:
//                   g (2 or 4 B) and p, m, v (4 B each) in, p, m, v out.
//                   Gradients are never written.
//
//  small_step_kernel -- both of the above in one launch for small lists: one
//                   thread-block cluster whose CTAs meet at the hardware
//                   cluster barrier between the square-sum and the update,
//                   with the same per-chunk code and the same fixed-order
//                   sum, hence the same bits.
//
// The kernels are HBM-bound streams (about 0.5 flop per byte); they use 16-
// and 32-byte vector accesses and no tensor cores.  Consecutive kernels of a
// step, and of consecutive steps, overlap by programmatic dependent launch:
// each kernel signals griddepcontrol.launch_dependents at its start, and the
// next one runs griddepcontrol.wait before it touches anything the previous
// one may write.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "soma_kernels.h"

namespace soma {
namespace {

// bf16 is the upper half of a binary32: widening is a shift / mask.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_one(uint16_t w) { return __uint_as_float((uint32_t)w << 16); }
// fp16 widens through CUDA's conversion.
__device__ __forceinline__ float2 f16_pair(uint32_t w) {
    __half2 h;
    memcpy(&h, &w, sizeof h);
    return __half22float2(h);
}
__device__ __forceinline__ float f16_one(uint16_t w) { return __half2float(__ushort_as_half(w)); }

// Two consecutive 16-bit elements of a 32-bit word (the lower one first).
template <int DT>
__device__ __forceinline__ float2 pair16(uint32_t w) {
    if (DT == kF16) return f16_pair(w);
    return make_float2(bf16_lo(w), bf16_hi(w));
}
template <int DT>
__device__ __forceinline__ float one16(uint16_t w) {
    return DT == kF16 ? f16_one(w) : bf16_one(w);
}

// Round two fp32 values to a packed pair of 16-bit values (nearest even).
template <int LOW>
__device__ __forceinline__ uint32_t pack16(float a, float b) {
    uint32_t w;
    if (LOW == kF16) {
        const __half2 h = __floats2half2_rn(a, b);
        memcpy(&w, &h, sizeof w);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        memcpy(&w, &h, sizeof w);
    }
    return w;
}
template <int LOW>
__device__ __forceinline__ uint16_t one_to16(float a) {
    return LOW == kF16 ? __half_as_ushort(__float2half_rn(a)) : __bfloat16_as_ushort(__float2bfloat16_rn(a));
}

// Copy the chunk's segment descriptors into shared memory (4 x 16 B each).
__device__ __forceinline__ int stage_segments(const Table& t, int chunk, Seg* sm) {
    constexpr int kWords = sizeof(Seg) / sizeof(uint4);
    const int b = __ldg(t.chunk_begin + chunk);
    const int n = __ldg(t.chunk_begin + chunk + 1) - b;
    const uint4* src = reinterpret_cast<const uint4*>(t.segs + b);
    uint4* dst = reinterpret_cast<uint4*>(sm);
    for (int i = threadIdx.x; i < kWords * n; i += blockDim.x) dst[i] = __ldg(src + i);
    __syncthreads();
    return n;
}

template <int BLOCK>
__device__ __forceinline__ float block_sum(float x, float* scratch) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) scratch[w] = x;
    __syncthreads();
    float r = 0.f;
    if (w == 0) {
        r = (l < BLOCK / 32) ? scratch[l] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    }
    return r;  // valid in thread 0
}

// fp64 block sum (valid in thread 0).  An fp64 add takes about 128 cycles
// on this GPU, so the second level runs only log2(BLOCK / 32) butterfly steps.
template <int BLOCK>
__device__ __forceinline__ double block_sum64(double x, double* scratch) {
    static_assert(BLOCK % 64 == 0 && ((BLOCK / 32) & (BLOCK / 32 - 1)) == 0, "power-of-two warp count");
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) scratch[w] = x;
    __syncthreads();
    double r = 0.0;
    if (w == 0) {
        r = (l < BLOCK / 32) ? scratch[l] : 0.0;
#pragma unroll
        for (int o = BLOCK / 64; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    }
    return r;
}

// min(1, max_norm / (norm + 1e-6)), NaN propagating.  The quotient is formed
// only when it can be below 1: when max_norm >= norm + 1e-6 it rounds to at
// least 1 anyway, and an fp64 division takes about 550 cycles on this GPU.
__device__ __forceinline__ double clip_coefficient(double norm, double max_norm) {
    const double x = norm + 1e-6;
    if (max_norm >= x) return 1.0;
    const double q = max_norm / x;  // NaN when norm is NaN
    return q < 1.0 ? q : (q == q ? 1.0 : q);
}

// Read-only 16-byte load of gradient words that this kernel reads once: not
// allocated in L1 (same-box A/B: the square-sum kernel 7 % faster on the
// action-expert list, 10 % on the 20 000-tensor list).
__device__ __forceinline__ uint4 ld_once(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---- square-sum of one segment, accumulated into a0 / a1 -----------------

template <int DT>
__device__ __forceinline__ void sq8_16(const uint4 w, float& a0, float& a1) {
    float2 x;
    x = pair16<DT>(w.x); a0 = fmaf(x.x, x.x, a0); a1 = fmaf(x.y, x.y, a1);
    x = pair16<DT>(w.y); a0 = fmaf(x.x, x.x, a0); a1 = fmaf(x.y, x.y, a1);
    x = pair16<DT>(w.z); a0 = fmaf(x.x, x.x, a0); a1 = fmaf(x.y, x.y, a1);
    x = pair16<DT>(w.w); a0 = fmaf(x.x, x.x, a0); a1 = fmaf(x.y, x.y, a1);
}

__device__ __forceinline__ void sq4_f32(const float4 u, float& a0, float& a1) {
    a0 = fmaf(u.x, u.x, a0); a1 = fmaf(u.y, u.y, a1);
    a0 = fmaf(u.z, u.z, a0); a1 = fmaf(u.w, u.w, a1);
}

// Exclusive prefix sums over the staged segments of a chunk (at most 64):
// upre[k] = 16-byte units of vector body in segments before k (one unit per
// 8-element vector of a 16-bit gradient, two for fp32), spre[k] = elements
// handled one at a time (head + tail) before k; upre[64] / spre[64] hold the
// totals.  One warp scans, two segments per lane.
// kUnits: count 16-byte units of gradient (square-sum); otherwise count
// 8-element vectors (update).
template <bool kUnits>
__device__ __forceinline__ int body_count(const Seg& s) {
    return (kUnits && s.gdtype == kF32) ? 2 * s.nvec : s.nvec;
}

// Is the vector body of s 32-byte aligned in p, m, v and, for fp32
// gradients, g?  (Every vector of the body then is.)
__device__ __forceinline__ bool wide_body(const Seg& s) {
    uintptr_t a = (uintptr_t)(s.p + s.head) | (uintptr_t)(s.m + s.head) | (uintptr_t)(s.v + s.head);
    if (s.gdtype == kF32) a |= (uintptr_t)(static_cast<const float*>(s.g) + s.head);
    return (a & 31) == 0;
}

template <bool kUnits>
__device__ __forceinline__ void segment_prefix(const Seg* segs, int ns, int* upre, int* spre) {
    static_assert(kMaxSegsPerChunk == 64, "two segments per lane");
    if (threadIdx.x < 32) {
        const unsigned full = 0xffffffffu;
        const int l = threadIdx.x;
        const int v0 = l < ns ? body_count<kUnits>(segs[l]) : 0;
        const int v1 = l + 32 < ns ? body_count<kUnits>(segs[l + 32]) : 0;
        const int s0 = l < ns ? segs[l].len - kVec * segs[l].nvec : 0;
        const int s1 = l + 32 < ns ? segs[l + 32].len - kVec * segs[l + 32].nvec : 0;
        int iv0 = v0, iv1 = v1, is0 = s0, is1 = s1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t;
            t = __shfl_up_sync(full, iv0, o); if (l >= o) iv0 += t;
            t = __shfl_up_sync(full, iv1, o); if (l >= o) iv1 += t;
            t = __shfl_up_sync(full, is0, o); if (l >= o) is0 += t;
            t = __shfl_up_sync(full, is1, o); if (l >= o) is1 += t;
        }
        const int tv0 = __shfl_sync(full, iv0, 31), ts0 = __shfl_sync(full, is0, 31);
        upre[l] = iv0 - v0;
        upre[l + 32] = tv0 + iv1 - v1;
        spre[l] = is0 - s0;
        spre[l + 32] = ts0 + is1 - s1;
        if (l == 31) {
            upre[64] = tv0 + iv1;
            spre[64] = ts0 + is1;
        }
    }
    __syncthreads();
}

// Square-sum of a chunk made of one segment: the gradient dtype is fixed at
// compile time and each thread walks units t, t + B, ... four at a time.
template <int DT>
__device__ __forceinline__ void segment_sumsq(const Seg& s, float& a0, float& a1) {
    const int B = blockDim.x;
    const int esize = DT == kF32 ? 4 : 2;
    const uint4* base = reinterpret_cast<const uint4*>(static_cast<const char*>(s.g) + s.head * esize);
    const int U = DT == kF32 ? 2 * s.nvec : s.nvec;
    int u = threadIdx.x;
    for (; u + 3 * B < U; u += 4 * B) {
        const uint4 w0 = ld_once(base + u), w1 = ld_once(base + u + B);
        const uint4 w2 = ld_once(base + u + 2 * B), w3 = ld_once(base + u + 3 * B);
        if (DT == kF32) {
            sq4_f32(make_float4(__uint_as_float(w0.x), __uint_as_float(w0.y), __uint_as_float(w0.z),
                                __uint_as_float(w0.w)), a0, a1);
            sq4_f32(make_float4(__uint_as_float(w1.x), __uint_as_float(w1.y), __uint_as_float(w1.z),
                                __uint_as_float(w1.w)), a0, a1);
            sq4_f32(make_float4(__uint_as_float(w2.x), __uint_as_float(w2.y), __uint_as_float(w2.z),
                                __uint_as_float(w2.w)), a0, a1);
            sq4_f32(make_float4(__uint_as_float(w3.x), __uint_as_float(w3.y), __uint_as_float(w3.z),
                                __uint_as_float(w3.w)), a0, a1);
        } else {
            sq8_16<DT>(w0, a0, a1);
            sq8_16<DT>(w1, a0, a1);
            sq8_16<DT>(w2, a0, a1);
            sq8_16<DT>(w3, a0, a1);
        }
    }
    for (; u < U; u += B) {
        const uint4 w = ld_once(base + u);
        if (DT == kF32)
            sq4_f32(make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                                __uint_as_float(w.w)), a0, a1);
        else
            sq8_16<DT>(w, a0, a1);
    }
    for (int j = threadIdx.x; j < s.len - kVec * s.nvec; j += B) {  // head, then tail
        const int idx = j < s.head ? j : s.head + kVec * s.nvec + (j - s.head);
        float x;
        if (DT == kF32) x = __ldg(static_cast<const float*>(s.g) + idx);
        else x = one16<DT>(__ldg(static_cast<const uint16_t*>(s.g) + idx));
        a1 = fmaf(x, x, a1);
    }
}

// Square-sum of one chunk.  The 16-byte units of all its segments' vector
// bodies form one index space; thread t takes units t, t + B, t + 2B, ...
// (B = block size), four loads in flight whatever the segment sizes, and
// follows its segment with a cursor that only moves forward.  The head and
// tail elements are flattened the same way.
__device__ __forceinline__ void chunk_sumsq(const Seg* segs, const int* upre, const int* spre, float& a0,
                                            float& a1) {
    const int B = blockDim.x;
    const int U = upre[kMaxSegsPerChunk];
    int k = 0;
    for (int u0 = threadIdx.x; u0 < U; u0 += 4 * B) {
        uint4 w[4];
        uint8_t dt[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int u = u0 + q * B;
            dt[q] = 0xff;
            if (u < U) {
                while (u >= upre[k + 1]) ++k;
                const Seg& sg = segs[k];
                dt[q] = sg.gdtype;
                const char* base = static_cast<const char*>(sg.g) + sg.head * (sg.gdtype == kF32 ? 4 : 2);
                w[q] = ld_once(reinterpret_cast<const uint4*>(base) + (u - upre[k]));
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (dt[q] == kF32) {
                sq4_f32(make_float4(__uint_as_float(w[q].x), __uint_as_float(w[q].y), __uint_as_float(w[q].z),
                                    __uint_as_float(w[q].w)), a0, a1);
            } else if (dt[q] == kBF16) {
                sq8_16<kBF16>(w[q], a0, a1);
            } else if (dt[q] == kF16) {
                sq8_16<kF16>(w[q], a0, a1);
            }
        }
    }
    const int S = spre[kMaxSegsPerChunk];
    k = 0;
    for (int e = threadIdx.x; e < S; e += B) {
        while (e >= spre[k + 1]) ++k;
        const Seg& sg = segs[k];
        const int j = e - spre[k];
        const int idx = j < sg.head ? j : sg.head + kVec * sg.nvec + (j - sg.head);
        float x;
        if (sg.gdtype == kF32) x = __ldg(static_cast<const float*>(sg.g) + idx);
        else if (sg.gdtype == kBF16) x = bf16_one(__ldg(static_cast<const uint16_t*>(sg.g) + idx));
        else x = f16_one(__ldg(static_cast<const uint16_t*>(sg.g) + idx));
        a1 = fmaf(x, x, a1);
    }
}

// Step constants of one group at step t: the same fp64 arithmetic, rounded
// the same way, as the host derivation of a regular step.
__device__ __noinline__ GroupHp group_constants(const DevGroup& g, int64_t t) {
    return make_group_hp(g.lr, g.beta1, g.beta2, g.eps, g.weight_decay, t);
}

// Square-sum of one staged norm chunk over the whole CTA (fp32 per-thread
// sums, then the fixed-shape block tree); the total is valid in thread 0.
__device__ __forceinline__ float chunk_square_sum(const Seg* segs, int ns, int* upre, int* spre, float* wsum) {
    float a0 = 0.f, a1 = 0.f;
    if (ns == 1) {
        if (segs[0].gdtype == kBF16) segment_sumsq<kBF16>(segs[0], a0, a1);
        else if (segs[0].gdtype == kF16) segment_sumsq<kF16>(segs[0], a0, a1);
        else segment_sumsq<kF32>(segs[0], a0, a1);
    } else {
        segment_prefix<true>(segs, ns, upre, spre);
        chunk_sumsq(segs, upre, spre, a0, a1);
    }
    return block_sum<kNormBlock>(a0 + a1, wsum);
}

// The n chunk partials added in one fixed order: thread t adds partials t,
// t + B, t + 2B, ... (B = block size), eight loads in flight at a time, then
// a fixed-shape block tree.  The total is valid in thread 0.
__device__ __forceinline__ double partials_sum(const double* partials, int n, double* wsum64) {
    double s = 0.0;
    const int B = blockDim.x;
    int i = threadIdx.x;
    for (; i + 7 * B < n; i += 8 * B) {
        double x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = __ldcg(partials + i + u * B);
        // pairwise: three dependent fp64 adds rather than eight
        s += ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
    }
    for (; i < n; i += B) s += __ldcg(partials + i);
    return block_sum64<kNormBlock>(s, wsum64);
}

// kGroupDiv: some group has its own divisor.  Each norm chunk then belongs to
// one group, and its partial is scaled by that group's 1/d^2; otherwise the
// partials are raw sums of g^2 and the step's d is applied to the total.
template <bool kGraph, bool kGroupDiv>
__global__ void __launch_bounds__(kNormBlock, 3) norm_kernel(const __grid_constant__ NormArgs a) {
    __shared__ __align__(16) Seg segs[kMaxSegsPerChunk];
    __shared__ int upre[kMaxSegsPerChunk + 1], spre[kMaxSegsPerChunk + 1];
    __shared__ float wsum[kNormBlock / 32];
    __shared__ double wsum64[kNormBlock / 32];
    __shared__ int last;

    // The update kernel may be scheduled as soon as every CTA of this one
    // has started; it waits for this grid's results before using them.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int first = kGraph ? (int)blockIdx.x - 1 : (int)blockIdx.x;
    const int stride = kGraph ? (int)gridDim.x - 1 : (int)gridDim.x;
    // This kernel itself may start before the preceding kernel on the stream
    // has finished (programmatic serialization): stage the first chunk's
    // segments (the tables only), then wait for that kernel before reading
    // any gradient or writing anything another kernel reads.
    const int ns0 = (first >= 0 && first < a.t.nchunks) ? stage_segments(a.t, first, segs) : 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Graph steps: CTA 0 advances the step counts and derives the group
    // constants (they do not depend on the norm), alongside the chunk CTAs
    // rather than after the reduction.
    if (kGraph && blockIdx.x == 0) {
        for (int q = threadIdx.x; q < a.ngroups && q < kMaxGroups; q += blockDim.x) {
            if ((a.present >> q) & 1ull) {
                const int64_t t = a.dgroups[q].step + 1;
                a.dgroups[q].step = t;
                a.dhp[q] = group_constants(a.dgroups[q], t);
            }
        }
    }
    for (int c = first; c >= 0 && c < a.t.nchunks; c += stride) {
        const int ns = c == first ? ns0 : stage_segments(a.t, c, segs);
        const float bs = chunk_square_sum(segs, ns, upre, spre, wsum);
        if (threadIdx.x == 0) {
            if (kGroupDiv) {
                const double w = a.inv_divisor[segs[0].group];
                a.partials[c] = (double)bs * w * w;
            } else {
                a.partials[c] = (double)bs;
            }
        }
        __syncthreads();  // segs and wsum are reused by the next chunk
    }

    // Arrival: the last CTA to finish reduces all partials.  No CTA waits.
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned t = atomicAdd(&a.res->ticket, 1u);
        last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();

    const double s = partials_sum(a.partials, a.t.nchunks, wsum64);
    if (threadIdx.x == 0) {
        const double norm = kGroupDiv ? sqrt(s) : sqrt(s) * a.inv_step_divisor;
        const double coef = clip_coefficient(norm, a.max_norm);
        a.res->sumsq = s;
        a.res->norm = norm;
        a.res->coef = coef;
        a.res->scale = (float)(coef * a.inv_step_divisor);
        a.res->nonfinite = isfinite(norm) ? 0u : 1u;
        // (a multi-rank step counts its global norm in the finish kernel)
        if (!isfinite(norm) && !a.sumsq_out) a.res->nonfinite_steps += 1u;
        a.res->ticket = 0u;
        if (a.sumsq_out) *a.sumsq_out = kGroupDiv ? s : s * a.inv_step_divisor * a.inv_step_divisor;
        wsum64[0] = coef;
    }
    if (kGroupDiv) {
        __syncthreads();
        const double coef = wsum64[0];
        for (int q = threadIdx.x; q < a.ngroups && q < kMaxGroups; q += blockDim.x)
            a.gscale[q] = (float)(coef * a.inv_divisor[q]);
    }
}

// Multi-rank step: the global norm from the ranks' square-sums, added in
// rank order so every rank derives the same bits.
__global__ void finish_kernel(const __grid_constant__ FinishArgs a) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    double s = 0.0;
    for (int r = 0; r < a.count; ++r) s += a.parts[r];
    const double norm = sqrt(s);
    const double coef = clip_coefficient(norm, a.max_norm);
    a.res->sumsq = s;
    a.res->norm = norm;
    a.res->coef = coef;
    a.res->scale = (float)(coef * a.inv_step_divisor);
    a.res->nonfinite = isfinite(norm) ? 0u : 1u;
    if (!isfinite(norm)) a.res->nonfinite_steps += 1u;
    if (a.gscale)
        for (int q = 0; q < a.ngroups && q < kMaxGroups; ++q) a.gscale[q] = (float)(coef * a.inv_divisor[q]);
}

// ---- fused update --------------------------------------------------------

__device__ __forceinline__ void adamw(float& p, float& m, float& v, float g, const GroupHp& h) {
    p *= h.decay;
    m = fmaf(h.beta1, m, h.one_minus_beta1 * g);
    v = fmaf(h.beta2, v, h.one_minus_beta2 * (g * g));
    const float denom = fmaf(sqrtf(v), h.inv_sqrt_bc2, h.eps);
    p = fmaf(-h.step_size, m / denom, p);
}

// One element j of a segment, any gradient and copy dtype.
__device__ __forceinline__ void update_one(const Seg& s, int j, const GroupHp& h, float scale) {
    float g;
    if (s.gdtype == kF32) g = __ldcs(static_cast<const float*>(s.g) + j);
    else if (s.gdtype == kBF16) g = bf16_one(__ldcs(static_cast<const unsigned short*>(s.g) + j));
    else g = f16_one(__ldcs(static_cast<const unsigned short*>(s.g) + j));
    float p = __ldcs(s.p + j), m = __ldcs(s.m + j), v = __ldcs(s.v + j);
    adamw(p, m, v, g * scale, h);
    __stcs(s.p + j, p);
    __stcs(s.m + j, m);
    __stcs(s.v + j, v);
    if (s.lowdt == kBF16) __stcs(static_cast<unsigned short*>(s.plow) + j, one_to16<kBF16>(p));
    else if (s.lowdt == kF16) __stcs(static_cast<unsigned short*>(s.plow) + j, one_to16<kF16>(p));
}

// Eight consecutive elements of the vector body: raw gradient words as
// loaded (one 16-byte word for 16-bit gradients, two for fp32) and p, m, v.
struct Lane8 {
    uint4 g0, g1;
    float4 p0, p1, m0, m1, v0, v1;
};

// 32-byte accesses (sm_100 and later): eight fp32 values, or the two
// 16-byte words of eight fp32 gradients, in one instruction.  The address
// must be 32-byte aligned; callers check that first.
__device__ __forceinline__ void ld32_f32(const float* p, float4& a, float4& b) {
    asm volatile("ld.global.cs.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(a.x), "=f"(a.y), "=f"(a.z), "=f"(a.w), "=f"(b.x), "=f"(b.y), "=f"(b.z), "=f"(b.w)
                 : "l"(p));
}
__device__ __forceinline__ void ld32_u32(const void* p, uint4& a, uint4& b) {
    asm volatile("ld.global.cs.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(p));
}
__device__ __forceinline__ void st32_f32(float* p, const float4& a, const float4& b) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"l"(p), "f"(a.x), "f"(a.y), "f"(a.z), "f"(a.w), "f"(b.x), "f"(b.y), "f"(b.z), "f"(b.w)
                 : "memory");
}


template <int DT>
__device__ __forceinline__ void load8_t(const Seg& s, int i, Lane8& x) {
    const float4* p = reinterpret_cast<const float4*>(s.p + s.head) + 2 * i;
    const float4* m = reinterpret_cast<const float4*>(s.m + s.head) + 2 * i;
    const float4* v = reinterpret_cast<const float4*>(s.v + s.head) + 2 * i;
    if (DT == kF32) {
        const uint4* g = reinterpret_cast<const uint4*>(static_cast<const float*>(s.g) + s.head) + 2 * i;
        x.g0 = __ldcs(g);
        x.g1 = __ldcs(g + 1);
    } else {
        x.g0 = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(s.g) + s.head) + i);
    }
    x.p0 = __ldcs(p); x.p1 = __ldcs(p + 1);
    x.m0 = __ldcs(m); x.m1 = __ldcs(m + 1);
    x.v0 = __ldcs(v); x.v1 = __ldcs(v + 1);
}

// Vector i of the body with 32-byte accesses (wide_body holds).
template <int DT>
__device__ __forceinline__ void load8_w(const Seg& s, int i, Lane8& x) {
    const int e = s.head + kVec * i;
    if (DT == kF32) ld32_u32(static_cast<const float*>(s.g) + e, x.g0, x.g1);
    else x.g0 = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(s.g) + s.head) + i);
    ld32_f32(s.p + e, x.p0, x.p1);
    ld32_f32(s.m + e, x.m0, x.m1);
    ld32_f32(s.v + e, x.v0, x.v1);
}

// Vector i of any segment: 32-byte accesses where its body allows them.
__device__ __forceinline__ void load8(const Seg& s, int i, Lane8& x) {
    const bool wide = wide_body(s);
    if (s.gdtype == kF32) {
        if (wide) load8_w<kF32>(s, i, x);
        else load8_t<kF32>(s, i, x);
    } else {  // one 16-byte word for either 16-bit type
        if (wide) load8_w<kBF16>(s, i, x);
        else load8_t<kBF16>(s, i, x);
    }
}

template <int DT>
__device__ __forceinline__ void widen8(const Lane8& x, float (&g)[8]) {
    if (DT == kF32) {
        g[0] = __uint_as_float(x.g0.x); g[1] = __uint_as_float(x.g0.y);
        g[2] = __uint_as_float(x.g0.z); g[3] = __uint_as_float(x.g0.w);
        g[4] = __uint_as_float(x.g1.x); g[5] = __uint_as_float(x.g1.y);
        g[6] = __uint_as_float(x.g1.z); g[7] = __uint_as_float(x.g1.w);
    } else {
        float2 t;
        t = pair16<DT>(x.g0.x); g[0] = t.x; g[1] = t.y;
        t = pair16<DT>(x.g0.y); g[2] = t.x; g[3] = t.y;
        t = pair16<DT>(x.g0.z); g[4] = t.x; g[5] = t.y;
        t = pair16<DT>(x.g0.w); g[6] = t.x; g[7] = t.y;
    }
}

template <int DT>
__device__ __forceinline__ void compute8_t(Lane8& x, const GroupHp& h, float scale) {
    float g[8];
    widen8<DT>(x, g);
    adamw(x.p0.x, x.m0.x, x.v0.x, g[0] * scale, h);
    adamw(x.p0.y, x.m0.y, x.v0.y, g[1] * scale, h);
    adamw(x.p0.z, x.m0.z, x.v0.z, g[2] * scale, h);
    adamw(x.p0.w, x.m0.w, x.v0.w, g[3] * scale, h);
    adamw(x.p1.x, x.m1.x, x.v1.x, g[4] * scale, h);
    adamw(x.p1.y, x.m1.y, x.v1.y, g[5] * scale, h);
    adamw(x.p1.z, x.m1.z, x.v1.z, g[6] * scale, h);
    adamw(x.p1.w, x.m1.w, x.v1.w, g[7] * scale, h);
}

__device__ __forceinline__ void compute8(const Seg& s, Lane8& x, const GroupHp& h, float scale) {
    if (s.gdtype == kF32) compute8_t<kF32>(x, h, scale);
    else if (s.gdtype == kBF16) compute8_t<kBF16>(x, h, scale);
    else compute8_t<kF16>(x, h, scale);
}

template <int LOW>
__device__ __forceinline__ uint4 pack8(const Lane8& x) {
    uint4 w;
    w.x = pack16<LOW>(x.p0.x, x.p0.y);
    w.y = pack16<LOW>(x.p0.z, x.p0.w);
    w.z = pack16<LOW>(x.p1.x, x.p1.y);
    w.w = pack16<LOW>(x.p1.z, x.p1.w);
    return w;
}

template <int LOW>
__device__ __forceinline__ void store8_t(const Seg& s, int i, const Lane8& x) {
    float4* p = reinterpret_cast<float4*>(s.p + s.head) + 2 * i;
    float4* m = reinterpret_cast<float4*>(s.m + s.head) + 2 * i;
    float4* v = reinterpret_cast<float4*>(s.v + s.head) + 2 * i;
    __stcs(p, x.p0); __stcs(p + 1, x.p1);
    __stcs(m, x.m0); __stcs(m + 1, x.m1);
    __stcs(v, x.v0); __stcs(v + 1, x.v1);
    if (LOW != kNone)
        __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(s.plow) + s.head) + i, pack8<LOW>(x));
}

template <int LOW>
__device__ __forceinline__ void store8_w(const Seg& s, int i, const Lane8& x) {
    const int e = s.head + kVec * i;
    st32_f32(s.p + e, x.p0, x.p1);
    st32_f32(s.m + e, x.m0, x.m1);
    st32_f32(s.v + e, x.v0, x.v1);
    if (LOW != kNone)
        __stcs(reinterpret_cast<uint4*>(static_cast<uint16_t*>(s.plow) + s.head) + i, pack8<LOW>(x));
}

__device__ __forceinline__ void store8(const Seg& s, int i, const Lane8& x) {
    if (wide_body(s)) {
        if (s.lowdt == kBF16) store8_w<kBF16>(s, i, x);
        else if (s.lowdt == kF16) store8_w<kF16>(s, i, x);
        else store8_w<kNone>(s, i, x);
    } else {
        if (s.lowdt == kBF16) store8_t<kBF16>(s, i, x);
        else if (s.lowdt == kF16) store8_t<kF16>(s, i, x);
        else store8_t<kNone>(s, i, x);
    }
}

// L2 prefetch of the gradient, p, m and v of this thread's first
// kPrefetchVectors vectors (all of an 8 Ki-element chunk, two thirds of a
// 12 Ki one; the sweep was taken with 16 Ki chunks).  Same-box sweep
// of 0-8: 4 was best on every list (the step 0.7 % faster than with 2 on the
// action-expert list, 0.6 % on the 7B shard view); 8 was up to 10 % slower.
constexpr int kPrefetchVectors = 4;

// The same for a chunk of several segments: this thread's first vectors of
// the chunk's flattened index space (vpre from segment_prefix).  Same-box
// A/B: the step 0.6 % faster on the 20 000-tensor list.
__device__ __forceinline__ void prefetch_flat(const Seg* segs, const int* vpre) {
    const int V = vpre[kMaxSegsPerChunk];
    int k = 0;
    for (int q = 0; q < kPrefetchVectors; ++q) {
        const int v = threadIdx.x + q * blockDim.x;
        if (v >= V) break;
        while (v >= vpre[k + 1]) ++k;
        const Seg& s = segs[k];
        const int e = s.head + kVec * (v - vpre[k]);
        const int gsz = s.gdtype == kF32 ? 4 : 2;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(s.g) + (size_t)e * gsz));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(s.p + e));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(s.m + e));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(s.v + e));
    }
}

// L2 prefetch of the gradient, p, m and v of vector i of segment s.
__device__ __forceinline__ void prefetch_vector(const Seg& s, int i) {
    const int e = s.head + kVec * i;
    const int gsz = s.gdtype == kF32 ? 4 : 2;
    asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(s.g) + (size_t)e * gsz));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(s.p + e));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(s.m + e));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(s.v + e));
}

__device__ __forceinline__ void prefetch_vectors(const Seg& s) {
    for (int i = threadIdx.x, n = 0; i < s.nvec && n < kPrefetchVectors; i += blockDim.x, ++n) prefetch_vector(s, i);
}

// A chunk made of one segment (a slice of a large tensor): dtypes fixed at
// compile time, two vectors in flight per thread.  With 16-bit gradients each
// thread also prefetches its next pair of vectors into L2 while it loads the
// current pair, which puts more requests in flight without holding registers.
// Same-box A/B: the step 0.54 % faster on the 7B shard view and 0.56 % on the
// action-expert list; with fp32 gradients it was 1 % slower on the flat list,
// so fp32 gradients go without.
template <int DT, int LOW>
__device__ __forceinline__ void segment_update(const Seg& s, const GroupHp& h, float scale) {
    for (int j = threadIdx.x; j < s.head; j += blockDim.x) update_one(s, j, h, scale);
    const int n = s.nvec, B = blockDim.x;
    int i = threadIdx.x;
    if (wide_body(s)) {  // same-box A/B: 1.3 % faster on the action-expert list, 1.7 % on the flat list
        for (; i + B < n; i += 2 * B) {
            Lane8 x0, x1;
            load8_w<DT>(s, i, x0);
            load8_w<DT>(s, i + B, x1);
            if (DT != kF32 && i + 3 * B < n) {
                prefetch_vector(s, i + 2 * B);
                prefetch_vector(s, i + 3 * B);
            }
            compute8_t<DT>(x0, h, scale);
            compute8_t<DT>(x1, h, scale);
            store8_w<LOW>(s, i, x0);
            store8_w<LOW>(s, i + B, x1);
        }
    }
    for (; i + B < n; i += 2 * B) {
        Lane8 x0, x1;
        load8_t<DT>(s, i, x0);
        load8_t<DT>(s, i + B, x1);
        compute8_t<DT>(x0, h, scale);
        compute8_t<DT>(x1, h, scale);
        store8_t<LOW>(s, i, x0);
        store8_t<LOW>(s, i + B, x1);
    }
    if (i < n) {
        Lane8 x0;
        load8_t<DT>(s, i, x0);
        compute8_t<DT>(x0, h, scale);
        store8_t<LOW>(s, i, x0);
    }
    for (int j = s.head + kVec * s.nvec + threadIdx.x; j < s.len; j += B) update_one(s, j, h, scale);
}

template <int DT>
__device__ __forceinline__ void segment_update_low(const Seg& s, const GroupHp& h, float scale) {
    if (s.lowdt == kBF16) segment_update<DT, kBF16>(s, h, scale);
    else if (s.lowdt == kF16) segment_update<DT, kF16>(s, h, scale);
    else segment_update<DT, kNone>(s, h, scale);
}

// One chunk of the update.  The 8-element vectors of all its segments form
// one index space; thread t takes vectors t, t + B, t + 2B, ... two at a
// time (both loaded before either is used), following its segment with a
// forward-only cursor, so small tensors keep as many loads in flight as
// large ones.  Head and tail elements are flattened the same way.
template <bool kGraph, bool kGroupDiv>
__device__ __forceinline__ void chunk_update(const Seg* segs, const int* vpre, const int* spre,
                                             const UpdateArgs& a, const GroupHp* shp, const float* gscale,
                                             float scale1) {
    auto scale_of = [&](const Seg& s) { return kGroupDiv ? gscale[s.group] : scale1; };
    const int B = blockDim.x;
    const int V = vpre[kMaxSegsPerChunk];
    int k = 0;
    for (int v0 = threadIdx.x; v0 < V; v0 += 2 * B) {
        Lane8 x0, x1;
        const int v1 = v0 + B;
        while (v0 >= vpre[k + 1]) ++k;
        const int k0 = k;
        load8(segs[k0], v0 - vpre[k0], x0);
        int k1 = -1;
        if (v1 < V) {
            while (v1 >= vpre[k + 1]) ++k;
            k1 = k;
            load8(segs[k1], v1 - vpre[k1], x1);
        }
        {
            const Seg& s = segs[k0];
            const GroupHp& h = kGraph ? shp[s.group] : a.groups[s.group];
            compute8(s, x0, h, scale_of(s));
            store8(s, v0 - vpre[k0], x0);
        }
        if (k1 >= 0) {
            const Seg& s = segs[k1];
            const GroupHp& h = kGraph ? shp[s.group] : a.groups[s.group];
            compute8(s, x1, h, scale_of(s));
            store8(s, v1 - vpre[k1], x1);
        }
    }
    const int S = spre[kMaxSegsPerChunk];
    k = 0;
    for (int e = threadIdx.x; e < S; e += B) {
        while (e >= spre[k + 1]) ++k;
        const Seg& s = segs[k];
        const int j = e - spre[k];
        const GroupHp& h = kGraph ? shp[s.group] : a.groups[s.group];
        update_one(s, j < s.head ? j : s.head + kVec * s.nvec + (j - s.head), h, scale_of(s));
    }
}

// Chunks run in reverse list order: the gradients the square-sum kernel read
// last are the ones most likely still in L2 when this kernel starts.
// kGroupDiv: some group sets its own divisor, so the scale c/d differs by
// group; otherwise every element uses the one scale the norm kernel wrote.
template <bool kGraph, bool kGroupDiv>
__global__ void __launch_bounds__(kUpdateBlock, 2) update_kernel(const __grid_constant__ UpdateArgs a) {
    // The next step's square-sum kernel may be scheduled once every CTA of
    // this one has started; it waits for this grid before reading gradients.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ __align__(16) Seg segs[kMaxSegsPerChunk];
    __shared__ int vpre[kMaxSegsPerChunk + 1], spre[kMaxSegsPerChunk + 1];
    __shared__ GroupHp shp[kGraph ? kMaxGroups : 1];
    __shared__ float gscale[kGroupDiv ? kMaxGroups : 1];  // c / d of each group
    float scale1 = 0.f;                                  // c / d when all groups share d
    bool ready = false, prefixed = false;  // prefixed: vpre/spre already hold this chunk's sums
    for (int r = blockIdx.x; r < a.t.nchunks; r += gridDim.x) {
        const int c = a.t.nchunks - 1 - r;
        const int ns = stage_segments(a.t, c, segs);
        if (!ready) {
            // Up to here only the tables and the caller's buffers were read, so
            // this can overlap the tail of the square-sum kernel (launched with
            // programmatic stream serialization).  Warm L2 with this thread's
            // first vectors, then wait for that kernel's results: the clip
            // scale and, for graph steps, the group constants.
            if (ns == 1) {
                prefetch_vectors(segs[0]);
            } else if (!kGraph) {  // (graph variants: more registers would spill)
                segment_prefix<false>(segs, ns, vpre, spre);
                prefetch_flat(segs, vpre);
                prefixed = true;
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            if (kGroupDiv) {
                for (int q = threadIdx.x; q < a.ngroups && q < kMaxGroups; q += blockDim.x)
                    gscale[q] = __ldcg(a.gscale + q);
            } else {
                scale1 = __ldcg(&a.res->scale);
            }
            if (kGraph) {
                for (int q = threadIdx.x; q < a.ngroups && q < kMaxGroups; q += blockDim.x) shp[q] = a.dhp[q];
            }
            if (kGraph || kGroupDiv) __syncthreads();
            ready = true;
        }
        if (ns == 1) {
            const Seg& s = segs[0];
            const GroupHp& h = kGraph ? shp[s.group] : a.groups[s.group];
            const float sc = kGroupDiv ? gscale[s.group] : scale1;
            if (s.gdtype == kBF16) segment_update_low<kBF16>(s, h, sc);
            else if (s.gdtype == kF16) segment_update_low<kF16>(s, h, sc);
            else segment_update_low<kF32>(s, h, sc);
        } else {
            if (!prefixed) segment_prefix<false>(segs, ns, vpre, spre);
            prefixed = false;
            chunk_update<kGraph, kGroupDiv>(segs, vpre, spre, a, shp, gscale, scale1);
        }
        __syncthreads();  // segs and the prefixes are rebuilt for the next chunk
    }
}

// Stages chunk ca of table ta into sa and chunk cb of tb into sb (a negative
// chunk: none) with the loads of both in flight together; returns the
// segment counts in na and nb.
__device__ __forceinline__ void stage_two(const Table& ta, int ca, Seg* sa, int& na, const Table& tb, int cb,
                                          Seg* sb, int& nb) {
    constexpr int kWords = sizeof(Seg) / sizeof(uint4);
    int ba = 0, ea = 0, bb = 0, eb = 0;
    if (ca >= 0) {
        ba = __ldg(ta.chunk_begin + ca);
        ea = __ldg(ta.chunk_begin + ca + 1);
    }
    if (cb >= 0) {
        bb = __ldg(tb.chunk_begin + cb);
        eb = __ldg(tb.chunk_begin + cb + 1);
    }
    na = ea - ba;
    nb = eb - bb;
    const uint4* srca = reinterpret_cast<const uint4*>(ta.segs + ba);
    const uint4* srcb = reinterpret_cast<const uint4*>(tb.segs + bb);
    uint4* dsta = reinterpret_cast<uint4*>(sa);
    uint4* dstb = reinterpret_cast<uint4*>(sb);
    for (int i = threadIdx.x; i < kWords * (na + nb); i += blockDim.x) {
        if (i < kWords * na) dsta[i] = __ldg(srca + i);
        else dstb[i - kWords * na] = __ldg(srcb + (i - kWords * na));
    }
    __syncthreads();
}

// partials_sum for n <= 32, in warp 0: the same total, because every term
// partials_sum adds beyond these 32 lanes' values is an exact +0 (each
// thread's sum starts at 0.0, and the other warps' sums are +0).
__device__ __forceinline__ double partials_sum_warp(const double* partials, int n) {
    double x = 0.0;
    if ((int)threadIdx.x < n) x = 0.0 + __ldcg(partials + threadIdx.x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// The whole step in one launch, for lists so small that the chain of two
// dependent kernels costs more than their work: one thread-block cluster of K
// CTAs (the grid is that one cluster).  CTA r square-sums norm chunks r,
// r + K, ... with the square-sum kernel's per-chunk code, so the partials are
// the same bits.  The hardware cluster barrier (release / acquire) then makes
// every partial visible to every CTA: no CTA polls memory.  Each CTA adds all
// partials in the square-sum kernel's fixed order, so all derive the same c
// and scale as that kernel's last CTA would; CTA 0 publishes norm and c.
// Then CTA r updates update chunks r, r + K, ... with the update kernel's
// per-element code.  The first update chunk's vectors, when there is at most
// one per thread, are loaded before the barrier: they do not depend on c.
// kGraph: the graph-capturable step; each CTA derives the group constants
// from the device group table (warp 1, while warp 0 adds the partials) from
// the step counts it read before the barrier, and CTA 0 writes the advanced
// counts back after it.  kGroupDiv: some group sets its own divisor; as in
// the two kernels, each partial is scaled by its chunk's group's 1/d^2 and
// every CTA forms c/d of each group.
template <bool kGraph, bool kGroupDiv>
__global__ void __launch_bounds__(kNormBlock, 1) small_step_kernel(const __grid_constant__ NormArgs na,
                                                                   const __grid_constant__ UpdateArgs ua) {
    __shared__ __align__(16) Seg segs[kMaxSegsPerChunk];   // norm chunk, later update chunks
    __shared__ __align__(16) Seg usegs[kMaxSegsPerChunk];  // the first update chunk
    __shared__ int upre[kMaxSegsPerChunk + 1], spre[kMaxSegsPerChunk + 1];
    __shared__ int vpre[kMaxSegsPerChunk + 1], vspre[kMaxSegsPerChunk + 1];
    __shared__ float wsum[kNormBlock / 32];
    __shared__ double wsum64[kNormBlock / 32];
    __shared__ GroupHp shp[kGraph ? kMaxGroups : 1];
    __shared__ float gs[kGroupDiv ? kMaxGroups : 1];  // c / d of each group

    // The next step's launch may be scheduled once every CTA has started; it
    // waits for this grid before touching anything.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int r = (int)blockIdx.x, K = (int)gridDim.x;
    const int warp = (int)threadIdx.x >> 5, lane = (int)threadIdx.x & 31;
    int ns0, nu0;
    stage_two(na.t, r < na.t.nchunks ? r : -1, segs, ns0, ua.t, r < ua.t.nchunks ? r : -1, usegs, nu0);
    asm volatile("griddepcontrol.wait;" ::: "memory");

    Lane8 x;
    int kx = -1;         // segment of this thread's early vector (vector index threadIdx.x), or none
    bool early = false;  // the first update chunk's vectors are loaded
    if (nu0 > 0) {
        segment_prefix<false>(usegs, nu0, vpre, vspre);
        const int V = vpre[kMaxSegsPerChunk];
        if (V <= (int)blockDim.x) {
            early = true;
            const int v = threadIdx.x;
            if (v < V) {
                int k = 0;
                while (v >= vpre[k + 1]) ++k;
                load8(usegs[k], v - vpre[k], x);
                kx = k;
            }
        }
    }

    // graph step: the step counts this step advances, read before the barrier
    // (CTA 0 writes the new ones after it); lane l of warp 1 holds groups l, l + 32
    int64_t t0 = 0, t1 = 0;
    if (kGraph && warp == 1) {
        if (lane < na.ngroups && ((na.present >> lane) & 1ull)) t0 = na.dgroups[lane].step + 1;
        if (lane + 32 < na.ngroups && ((na.present >> (lane + 32)) & 1ull)) t1 = na.dgroups[lane + 32].step + 1;
    }

    for (int c = r; c < na.t.nchunks; c += K) {
        const int ns = c == r ? ns0 : stage_segments(na.t, c, segs);
        const float bs = chunk_square_sum(segs, ns, upre, spre, wsum);
        if (threadIdx.x == 0) {
            if (kGroupDiv) {
                const double w = na.inv_divisor[segs[0].group];
                na.partials[c] = (double)bs * w * w;
            } else {
                na.partials[c] = (double)bs;
            }
        }
        __syncthreads();  // segs and wsum are reused by the next chunk
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");

    double s = 0.0;
    if (na.t.nchunks <= 32) {
        if (threadIdx.x < 32) s = partials_sum_warp(na.partials, na.t.nchunks);
    } else {
        s = partials_sum(na.partials, na.t.nchunks, wsum64);
    }
    if (kGraph && warp == 1) {
        if (t0 > 0) {
            shp[lane] = group_constants(na.dgroups[lane], t0);
            if (r == 0) na.dgroups[lane].step = t0;
        }
        if (t1 > 0) {
            shp[lane + 32] = group_constants(na.dgroups[lane + 32], t1);
            if (r == 0) na.dgroups[lane + 32].step = t1;
        }
    }
    if (threadIdx.x == 0) {
        const double norm = kGroupDiv ? sqrt(s) : sqrt(s) * na.inv_step_divisor;
        const double coef = clip_coefficient(norm, na.max_norm);
        const float scale = (float)(coef * na.inv_step_divisor);
        if (r == 0) {
            na.res->sumsq = s;
            na.res->norm = norm;
            na.res->coef = coef;
            na.res->scale = scale;
            na.res->nonfinite = isfinite(norm) ? 0u : 1u;
            if (!isfinite(norm)) na.res->nonfinite_steps += 1u;
        }
        wsum[0] = scale;
        wsum64[0] = coef;
    }
    __syncthreads();
    const float scale = wsum[0];
    if (kGroupDiv) {
        const double coef = wsum64[0];
        for (int q = threadIdx.x; q < na.ngroups && q < kMaxGroups; q += blockDim.x)
            gs[q] = (float)(coef * na.inv_divisor[q]);
        __syncthreads();
    }

    int c0 = r;
    if (early) {
        if (kx >= 0) {
            const Seg& sg = usegs[kx];
            compute8(sg, x, kGraph ? shp[sg.group] : ua.groups[sg.group], kGroupDiv ? gs[sg.group] : scale);
            store8(sg, (int)threadIdx.x - vpre[kx], x);
        }
        const int S = vspre[kMaxSegsPerChunk];
        int k = 0;
        for (int e = threadIdx.x; e < S; e += blockDim.x) {
            while (e >= vspre[k + 1]) ++k;
            const Seg& sg = usegs[k];
            const int j = e - vspre[k];
            update_one(sg, j < sg.head ? j : sg.head + kVec * sg.nvec + (j - sg.head),
                       kGraph ? shp[sg.group] : ua.groups[sg.group], kGroupDiv ? gs[sg.group] : scale);
        }
        c0 = r + K;
    }
    for (int c = c0; c < ua.t.nchunks; c += K) {
        const int ns = stage_segments(ua.t, c, segs);
        if (ns == 1) {
            const Seg& sg = segs[0];
            const GroupHp& h = kGraph ? shp[sg.group] : ua.groups[sg.group];
            const float sc = kGroupDiv ? gs[sg.group] : scale;
            if (sg.gdtype == kBF16) segment_update_low<kBF16>(sg, h, sc);
            else if (sg.gdtype == kF16) segment_update_low<kF16>(sg, h, sc);
            else segment_update_low<kF32>(sg, h, sc);
        } else {
            segment_prefix<false>(segs, ns, upre, spre);
            chunk_update<kGraph, kGroupDiv>(segs, upre, spre, ua, shp, gs, scale);
        }
        __syncthreads();  // segs and the prefixes are rebuilt for the next chunk
    }
}

}  // namespace

int launch_norm(const NormArgs& a, int grid, void* stream, bool graph, bool group_div, bool overlap) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kNormBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    cudaError_t e;
    if (graph && group_div) e = cudaLaunchKernelEx(&cfg, norm_kernel<true, true>, a);
    else if (graph) e = cudaLaunchKernelEx(&cfg, norm_kernel<true, false>, a);
    else if (group_div) e = cudaLaunchKernelEx(&cfg, norm_kernel<false, true>, a);
    else e = cudaLaunchKernelEx(&cfg, norm_kernel<false, false>, a);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

int launch_update(const UpdateArgs& a, int grid, void* stream, bool graph, bool overlap, bool group_div) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kUpdateBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    cudaError_t e;
    if (graph && group_div) e = cudaLaunchKernelEx(&cfg, update_kernel<true, true>, a);
    else if (graph) e = cudaLaunchKernelEx(&cfg, update_kernel<true, false>, a);
    else if (group_div) e = cudaLaunchKernelEx(&cfg, update_kernel<false, true>, a);
    else e = cudaLaunchKernelEx(&cfg, update_kernel<false, false>, a);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

int small_step_cluster_size() {
    const void* variants[4] = {reinterpret_cast<const void*>(small_step_kernel<false, false>),
                               reinterpret_cast<const void*>(small_step_kernel<false, true>),
                               reinterpret_cast<const void*>(small_step_kernel<true, false>),
                               reinterpret_cast<const void*>(small_step_kernel<true, true>)};
    for (const void* f : variants)
        if (cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
            (void)cudaGetLastError();
    for (int k = kSmallStepMaxCtas; k >= 2; k /= 2) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(k);
        cfg.blockDim = dim3(kNormBlock);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = k;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        bool all = true;
        for (const void* f : variants) {
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, f, &cfg) != cudaSuccess || clusters <= 0) all = false;
        }
        if (all) return k;
        (void)cudaGetLastError();
    }
    return 0;
}

int launch_small_step(const NormArgs& na, const UpdateArgs& ua, int ctas, void* stream, bool overlap, bool graph,
                      bool group_div) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kNormBlock);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 2 : 1;
    cudaError_t e;
    if (graph && group_div) e = cudaLaunchKernelEx(&cfg, small_step_kernel<true, true>, na, ua);
    else if (graph) e = cudaLaunchKernelEx(&cfg, small_step_kernel<true, false>, na, ua);
    else if (group_div) e = cudaLaunchKernelEx(&cfg, small_step_kernel<false, true>, na, ua);
    else e = cudaLaunchKernelEx(&cfg, small_step_kernel<false, false>, na, ua);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

int launch_finish(const FinishArgs& a, void* stream) {
    finish_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return (int)cudaGetLastError();
}

}  // namespace soma
