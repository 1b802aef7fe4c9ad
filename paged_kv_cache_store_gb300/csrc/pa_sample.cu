// pa_sample.cu -- Gumbel-max sampling of one token per row.
//
// What it computes [NV12 §12.2 "采样器": Sampler.forward and its Gumbel-max
// derivation]: for row b,
//     token[b] = argmax_i softmax(float(logits[b]) / T_b)_i / max(E[b, i], 1e-10)
// with E[b, i] ~ Exp(1) drawn independently per entry by the caller, in fp32;
// among equal maxima the lowest index wins (first maximum).
//
// How (GB300 design): the page's own derivation turns the division by E into
// a subtraction of log E under the argmax; with the softmax normaliser (one
// positive number per row) dropped as well, the token is the argmax of
//     key_i = logit_i * log2(e) / T - log2(max(E_i, 1e-10)),
// which orders the entries exactly as p_i / E_i does (log2 is increasing).
// So each thread keeps only its best (key, index): one lg2 and one fma per
// element, no running max and no rescaling.  Partial results combine by max
// key (lower index on equal keys) across a warp (shuffles), a CTA (shared
// memory) and the CTAs of a thread-block cluster that splits the row
// (distributed shared memory, into the cluster's first CTA).  One pass over
// HBM: every logit (2 or 4 bytes) and every draw (4 bytes) is read once with
// 16-byte loads.
#include <math.h>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int SAMPLE_THREADS = 256;
constexpr unsigned FULLM = 0xffffffffu;
constexpr float E_MIN = 1e-10f;  // the page's clamp of the exponential draws
#ifndef SAMPLE_MAX_CLUSTER
#define SAMPLE_MAX_CLUSTER 8
#endif
constexpr int MAX_CLUSTER = SAMPLE_MAX_CLUSTER;  // CTAs per row (a cluster)

// Partial argmax of a row: best key and its index (-inf and INT_MAX when
// nothing finite was seen; NaN keys never win).
struct __align__(8) Best {  // 8 bytes: one vector store into the cluster's first CTA
    float key;
    int idx;
};

__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ Best combine(Best a, Best b) { return better(b.key, b.idx, a.key, a.idx) ? b : a; }

__device__ __forceinline__ float key_of(float logit, float k, float e) {
    return fmaf(logit, k, -__log2f(fmaxf(e, E_MIN)));
}

// Read-once streaming loads (no L1 allocation).
__device__ __forceinline__ float4 ldg_stream(const float4 *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ldg_stream_u4(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <bool FP32>
__global__ void __launch_bounds__(SAMPLE_THREADS) sample_gumbel_kernel(
    int32_t *__restrict__ out, const void *__restrict__ logits, int64_t logits_stride,
    const float *__restrict__ temperatures, const float *__restrict__ noise, int64_t noise_stride, int32_t vocab,
    DevError *err) {
    pdl_wait_then_release();
    __shared__ Best part[SAMPLE_THREADS / 32];
    __shared__ Best cl[MAX_CLUSTER];  // used in the cluster's first CTA
    const int b = blockIdx.y;
    const uint32_t S = gridDim.x, rank = blockIdx.x;  // cluster = the S CTAs of a row
    const float T = __ldg(temperatures + b);
    const bool bad_t = !(T > 1e-10f);
    const float k = bad_t ? 0.f : 1.4426950408889634f / T;
    // This CTA's chunk of the row, a multiple of 8 elements except at the end.
    const int chunk = ((vocab + (int)S - 1) / (int)S + 7) & ~7;
    const int lo = min(vocab, (int)rank * chunk), hi = min(vocab, lo + chunk);
    Best s = {-INFINITY, 0x7fffffff};
    if (!bad_t) {
        const float *er = noise + (int64_t)b * noise_stride;
        const int nvec = (hi - lo) / 8;
        // Two 8-element groups per step, all loads issued first (48 bytes
        // each in flight per thread).
        for (int v0 = threadIdx.x; v0 < nvec; v0 += 2 * SAMPLE_THREADS) {
            float x[2][8], e[2][8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = v0 + h * SAMPLE_THREADS;
                const int i = lo + min(v, nvec - 1) * 8;  // a duplicate group past the end is ignored below
                const float4 e0 = ldg_stream(reinterpret_cast<const float4 *>(er + i));
                const float4 e1 = ldg_stream(reinterpret_cast<const float4 *>(er + i + 4));
                e[h][0] = e0.x; e[h][1] = e0.y; e[h][2] = e0.z; e[h][3] = e0.w;
                e[h][4] = e1.x; e[h][5] = e1.y; e[h][6] = e1.z; e[h][7] = e1.w;
                if (FP32) {
                    const float *lr = static_cast<const float *>(logits) + (int64_t)b * logits_stride;
                    const float4 a0 = ldg_stream(reinterpret_cast<const float4 *>(lr + i));
                    const float4 a1 = ldg_stream(reinterpret_cast<const float4 *>(lr + i + 4));
                    x[h][0] = a0.x; x[h][1] = a0.y; x[h][2] = a0.z; x[h][3] = a0.w;
                    x[h][4] = a1.x; x[h][5] = a1.y; x[h][6] = a1.z; x[h][7] = a1.w;
                } else {
                    const uint16_t *lr = static_cast<const uint16_t *>(logits) + (int64_t)b * logits_stride;
                    const uint4 w = ldg_stream_u4(reinterpret_cast<const uint4 *>(lr + i));
                    x[h][0] = bf16_lo(w.x); x[h][1] = bf16_hi(w.x); x[h][2] = bf16_lo(w.y); x[h][3] = bf16_hi(w.y);
                    x[h][4] = bf16_lo(w.z); x[h][5] = bf16_hi(w.z); x[h][6] = bf16_lo(w.w); x[h][7] = bf16_hi(w.w);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int v = v0 + h * SAMPLE_THREADS;
                if (v >= nvec) break;
                const int i = lo + v * 8;
                // The 8 keys are independent; a tree picks the best (lowest
                // index among equals), then it is merged into the running best.
                float kk[8];
                int ii[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    kk[j] = key_of(x[h][j], k, e[h][j]);
                    ii[j] = i + j;
                }
#pragma unroll
                for (int w = 1; w < 8; w <<= 1)
#pragma unroll
                    for (int j = 0; j < 8; j += 2 * w)
                        if (better(kk[j + w], ii[j + w], kk[j], ii[j])) {
                            kk[j] = kk[j + w];
                            ii[j] = ii[j + w];
                        }
                if (better(kk[0], ii[0], s.key, s.idx)) {
                    s.key = kk[0];
                    s.idx = ii[0];
                }
            }
        }
        for (int i = lo + nvec * 8 + threadIdx.x; i < hi; i += SAMPLE_THREADS) {  // ragged end of the row
            float x;
            if (FP32) {
                x = static_cast<const float *>(logits)[(int64_t)b * logits_stride + i];
            } else {
                const uint16_t h = static_cast<const uint16_t *>(logits)[(int64_t)b * logits_stride + i];
                x = __uint_as_float((uint32_t)h << 16);
            }
            const float kx = key_of(x, k, er[i]);
            if (better(kx, i, s.key, s.idx)) {
                s.key = kx;
                s.idx = i;
            }
        }
    }
    // Warp, then CTA.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Best t;
        t.key = __shfl_xor_sync(FULLM, s.key, o);
        t.idx = __shfl_xor_sync(FULLM, s.idx, o);
        s = combine(s, t);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < SAMPLE_THREADS / 32; ++w) s = combine(s, part[w]);
        // Into slot `rank` of the cluster's first CTA.
        uint32_t dst;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(smem_addr(&cl[rank])), "r"(0u));
        asm volatile("st.shared::cluster.v2.b32 [%0], {%1, %2};" ::"r"(dst), "r"(__float_as_uint(s.key)),
                     "r"((uint32_t)s.idx)
                     : "memory");
    }
    // Every thread of every CTA of the cluster arrives; the first CTA then
    // reads the slots (the others never touch shared memory again).
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (rank == 0 && threadIdx.x == 0) {
        Best r = cl[0];
        for (uint32_t c = 1; c < S; ++c) r = combine(r, cl[c]);
        if (bad_t) {
            record_error(err, PA_DEV_BAD_TEMPERATURE, b);
            out[b] = -1;
        } else {
            out[b] = (r.idx == 0x7fffffff) ? 0 : r.idx;  // no finite candidate: index 0
        }
    }
}

// CTAs per row: the smallest power of two that gives ~4 CTAs per SM over the
// batch, at most 8 (a portable cluster) and at least 2048 elements per CTA.
int ctas_per_row(int batch, int vocab, int sms) {
    int S = 1;
    while (S < MAX_CLUSTER && (int64_t)batch * S < 4LL * sms && vocab / (2 * S) >= 2048) S *= 2;
    return S;
}

template <bool FP32>
pa_status launch_sample(int32_t *out, const void *logits, int64_t logits_stride, const float *temperatures,
                        const float *noise, int64_t noise_stride, int32_t batch, int32_t vocab,
                        cudaStream_t stream) {
    const int S = ctas_per_row(batch, vocab, sm_count());
    if (MAX_CLUSTER > 8) {
        static bool done = false;
        if (!done) {
            cudaFuncSetAttribute(sample_gumbel_kernel<FP32>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            done = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)S, (unsigned)batch);
    cfg.blockDim = dim3(SAMPLE_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, sample_gumbel_kernel<FP32>, out, logits, logits_stride,
                                             temperatures, noise, noise_stride, vocab, device_error_ptr());
    if (e != cudaSuccess) return cuda_fail(e, "sample_gumbel_kernel");
    return check_launch("sample_gumbel_kernel");
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_sample_gumbel(int32_t *out_tokens, const void *logits, int64_t logits_row_stride,
                                      int32_t logits_is_fp32, const float *temperatures, const float *exp_noise,
                                      int64_t noise_row_stride, int32_t batch, int32_t vocab,
                                      pa_stream_t stream) {
    using namespace pa;
    if (batch < 0 || vocab < 0) return fail(PA_ERR_INVALID_ARG, "negative size");
    if (batch == 0) return PA_OK;
    if (vocab == 0) return fail(PA_ERR_INVALID_ARG, "vocab must be positive");
    if (batch > 65535) return fail(PA_ERR_UNSUPPORTED, "batch %d (at most 65535 rows per call)", batch);
    if (!out_tokens || !logits || !temperatures || !exp_noise) return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (logits_is_fp32 != 0 && logits_is_fp32 != 1) return fail(PA_ERR_INVALID_ARG, "logits_is_fp32 must be 0 or 1");
    const int align = logits_is_fp32 ? 4 : 8;  // elements per 16 bytes
    if (logits_row_stride < vocab || logits_row_stride % align)
        return fail(PA_ERR_INVALID_ARG, "logits_row_stride must be >= vocab and a multiple of %d", align);
    if (noise_row_stride < vocab || noise_row_stride % 4)
        return fail(PA_ERR_INVALID_ARG, "noise_row_stride must be >= vocab and a multiple of 4");
    if (!aligned16(logits) || !aligned16(exp_noise))
        return fail(PA_ERR_INVALID_ARG, "logits and exp_noise must be 16-byte aligned");
    if (sm_count() <= 0) return fail(PA_ERR_CUDA, "no CUDA device");
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return logits_is_fp32 ? launch_sample<true>(out_tokens, logits, logits_row_stride, temperatures, exp_noise,
                                                noise_row_stride, batch, vocab, s)
                          : launch_sample<false>(out_tokens, logits, logits_row_stride, temperatures, exp_noise,
                                                 noise_row_stride, batch, vocab, s);
}
