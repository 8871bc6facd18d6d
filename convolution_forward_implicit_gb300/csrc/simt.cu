// SIMT (FFMA) implicit-GEMM convolution forward for fp32 I/O, and for bf16 problems
// whose channel counts rule out the 16-byte tensor-core gather.  The arithmetic is fp32
// fused multiply-add throughout: no TF32, so fp32 I/O keeps fp32 products.
//
// Same GEMM view as the tensor-core kernel (page "composable_kernel ...
// LEARNINGS_GROUPED_CONV.md", introduction): per group, rows are output pixels, columns
// output channels, the reduction index kk = tap*C + c.  The activation tile is gathered
// from the channels-last input with zero fill in the padding (the implicit form of the
// im2col step on page "[ET-VK] conv1d runs at ~3% ...", section "The conv2d path already
// solves this"); the weight tile comes from the prepacked [G][taps*C][Kpad] matrix.
//
// CTA tile BM x 128 (BM = 128 or 64), K step 8, 256 threads, each thread an
// (BM/16) x 8 register block; double-buffered shared memory with register prefetch.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gelu.cuh"
#include "internal.h"

namespace convfwd {
namespace {

constexpr int BN = 128;
constexpr int BK = 8;
constexpr int THREADS = 256;

template <typename T> struct Io;
template <> struct Io<float> {
    static __device__ __forceinline__ float4 ld4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
    static __device__ __forceinline__ float ld1(const float* p) { return __ldg(p); }
    static __device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
        *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
    }
    static __device__ __forceinline__ void st1(float* p, float a) { *p = a; }
};
template <> struct Io<__nv_bfloat16> {
    static __device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    }
    static __device__ __forceinline__ float ld1(const __nv_bfloat16* p) { return __bfloat162float(p[0]); }
    static __device__ __forceinline__ void st4(__nv_bfloat16* p, float a, float b, float c, float d) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&lo);
        u.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p) = u;
    }
    static __device__ __forceinline__ void st1(__nv_bfloat16* p, float a) { p[0] = __float2bfloat16_rn(a); }
};


// Input offset of reduction index kk for a pixel, or -1 where the tap is in the padding.
struct PixelBase {
    int n, d0, h0, w0;   // n < 0 marks a row beyond M
};

// Backward data: the dy offset that tap `tap` draws on for an input pixel (pb holds its
// coordinates plus the padding), or -1 where no output position maps onto it.
__device__ __forceinline__ int src_pos(int num, int s, int O) {
    if (num < 0) return -1;
    const int o = num / s;
    return (o * s == num && o < O) ? o : -1;
}

__device__ __forceinline__ long long dy_offset(const Geom& g, const PixelBase& pb, int tap, int k, int gi) {
    if (pb.n < 0) return -1;
    const int yx = g.Y * g.X;
    const int z = tap / yx;
    const int r = tap - z * yx;
    const int y = r / g.X;
    const int x = r - y * g.X;
    const int od = src_pos(pb.d0 - z * g.dd, g.sd, g.Do);
    const int oh = src_pos(pb.h0 - y * g.dh, g.sh, g.Ho);
    const int ow = src_pos(pb.w0 - x * g.dw, g.sw, g.Wo);
    if ((od | oh | ow) < 0) return -1;
    return ((((long long)pb.n * g.Do + od) * g.Ho + oh) * g.Wo + ow) * (long long)(g.G * g.K) + (long long)gi * g.K + k;
}

__device__ __forceinline__ long long x_offset(const Geom& g, const PixelBase& pb, int tap, int c, int gi) {
    if (pb.n < 0) return -1;
    const int yx = g.Y * g.X;
    const int z = tap / yx;
    const int r = tap - z * yx;
    const int y = r / g.X;
    const int x = r - y * g.X;
    const int id = pb.d0 + z * g.dd, ih = pb.h0 + y * g.dh, iw = pb.w0 + x * g.dw;
    if ((unsigned)id >= (unsigned)g.D || (unsigned)ih >= (unsigned)g.H || (unsigned)iw >= (unsigned)g.W) return -1;
    return ((((long long)pb.n * g.D + id) * g.H + ih) * g.W + iw) * (long long)(g.G * g.C) + (long long)gi * g.C + c;
}

template <typename T, int BM, bool VEC, bool DG>
__global__ void __launch_bounds__(THREADS) conv_fwd_simt_kernel(const __grid_constant__ SimtParams p) {
    if (p.pdl) {   // a programmatic dependent: let the next kernel start, wait for the previous one
        griddep_launch();
        griddep_wait();
    }
    constexpr int TM = BM / 16;                 // rows per thread
    constexpr int A_LOADERS = BM * 2;           // threads that each load 4 consecutive kk of one row
    __shared__ __align__(16) float As[2][BK][BM + 4];
    __shared__ __align__(16) float Bs[2][BK][BN];

    const Geom& g = p.g;
    const T* x = reinterpret_cast<const T*>(p.x);
    const T* wpk = reinterpret_cast<const T*>(p.wpack);
    const int tid = threadIdx.x;
    const int mt = blockIdx.x, nt = blockIdx.y;
    const int gi = blockIdx.z / p.splits, split = blockIdx.z % p.splits;
    const int kt0 = split * p.ktps;
    const int kt1 = min(kt0 + p.ktps, p.nkt);

    // this thread's A row (pixel) and its base input coordinates
    const bool a_loader = tid < A_LOADERS;
    const int a_row = tid >> 1;
    const int a_kq = (tid & 1) * 4;
    PixelBase pb{-1, 0, 0, 0};
    if (a_loader) {
        const int m = mt * BM + a_row;
        if (m < p.rows) {
            int t = m;
            if (DG) {   // an input pixel; its coordinates plus the padding
                const int iw = t % g.W; t /= g.W;
                const int ih = t % g.H; t /= g.H;
                const int id = t % g.D;
                pb.n = t / g.D;
                pb.d0 = id + g.pd;
                pb.h0 = ih + g.ph;
                pb.w0 = iw + g.pw;
            } else {
                const int ow = t % g.Wo; t /= g.Wo;
                const int oh = t % g.Ho; t /= g.Ho;
                const int od = t % g.Do;
                pb.n = t / g.Do;
                pb.d0 = od * g.sd - g.pd;
                pb.h0 = oh * g.sh - g.ph;
                pb.w0 = ow * g.sw - g.pw;
            }
        }
    }
    // this thread's B slot
    const int b_k = tid >> 5;
    const int b_n = (tid & 31) * 4;
    const T* wg = wpk + (size_t)gi * p.Kg * p.Kpad + (size_t)nt * BN + b_n;

    float4 ra = make_float4(0.f, 0.f, 0.f, 0.f), rb;
    auto load_tile = [&](int kt) {
        const int kk0 = kt * BK;
        if (a_loader) {
            float v[4] = {0.f, 0.f, 0.f, 0.f};
            const int kk = kk0 + a_kq;
            if (VEC) {
                if (kk < p.Kg) {
                    const int tap = kk / p.rch;
                    const long long off = DG ? dy_offset(g, pb, tap, kk - tap * p.rch, gi)
                                             : x_offset(g, pb, tap, kk - tap * p.rch, gi);
                    if (off >= 0) {
                        const float4 f = Io<T>::ld4(x + off);
                        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k2 = kk + e;
                    if (k2 < p.Kg) {
                        const int tap = k2 / p.rch;
                        const long long off = DG ? dy_offset(g, pb, tap, k2 - tap * p.rch, gi)
                                                 : x_offset(g, pb, tap, k2 - tap * p.rch, gi);
                        if (off >= 0) v[e] = Io<T>::ld1(x + off);
                    }
                }
            }
            ra = make_float4(v[0], v[1], v[2], v[3]);
        }
        const int kb = kk0 + b_k;
        rb = (kb < p.Kg) ? Io<T>::ld4(wg + (size_t)kb * p.Kpad) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto store_tile = [&](int buf) {
        if (a_loader) {
            As[buf][a_kq + 0][a_row] = ra.x;
            As[buf][a_kq + 1][a_row] = ra.y;
            As[buf][a_kq + 2][a_row] = ra.z;
            As[buf][a_kq + 3][a_row] = ra.w;
        }
        *reinterpret_cast<float4*>(&Bs[buf][b_k][b_n]) = rb;
    };

    float acc[TM][8];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    const int tx = tid & 15, ty = tid >> 4;
    if (kt0 < kt1) {
        load_tile(kt0);
        store_tile(0);
        __syncthreads();
        for (int kt = kt0; kt < kt1; ++kt) {
            const int buf = (kt - kt0) & 1;
            if (kt + 1 < kt1) load_tile(kt + 1);
#pragma unroll
            for (int k = 0; k < BK; ++k) {
                float a[TM], b[8];
#pragma unroll
                for (int i = 0; i < TM; i += 4) {
                    const float4 t = *reinterpret_cast<const float4*>(&As[buf][k][ty * TM + i]);
                    a[i] = t.x; a[i + 1] = t.y; a[i + 2] = t.z; a[i + 3] = t.w;
                }
                const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][tx * 4]);
                const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][64 + tx * 4]);
                b[0] = b0.x; b[1] = b0.y; b[2] = b0.z; b[3] = b0.w;
                b[4] = b1.x; b[5] = b1.y; b[6] = b1.z; b[7] = b1.w;
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            if (kt + 1 < kt1) store_tile(buf ^ 1);
            __syncthreads();
        }
    }

    // epilogue
    T* y = reinterpret_cast<T*>(p.y);
    const T* bias = reinterpret_cast<const T*>(p.bias);
    const int NC = p.cols;
    const int GK = g.G * NC;
    const bool add_bias = !DG && (p.epi == EPI_BIAS || p.epi == EPI_BIAS_GELU) && p.splits == 1;
    const bool do_gelu = !DG && (p.epi == EPI_BIAS_GELU || p.epi == EPI_GELU) && p.splits == 1;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int m = mt * BM + ty * TM + i;
        if (m >= p.rows) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = nt * BN + h * 64 + tx * 4;
            if (n >= NC) continue;
            float v[4] = {acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]};
            const size_t o = (size_t)m * GK + (size_t)gi * NC + n;
            if (p.splits > 1) {
                float* dst = p.ws + (size_t)split * p.rows * GK + o;
                if (VEC) {
                    *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
                    for (int e = 0; e < 4 && n + e < NC; ++e) dst[e] = v[e];
                }
                continue;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (add_bias && n + e < NC) v[e] += Io<T>::ld1(bias + (size_t)gi * NC + n + e);
                if (do_gelu) v[e] = gelu(v[e]);
            }
            if (VEC) {
                Io<T>::st4(y + o, v[0], v[1], v[2], v[3]);
            } else {
                for (int e = 0; e < 4 && n + e < NC; ++e) Io<T>::st1(y + o + e, v[e]);
            }
        }
    }
}

template <typename T, int BM, bool VEC>
cudaError_t launch_t(const SimtParams& p, cudaStream_t stream) {
    dim3 grid(p.num_mt, p.num_nt, p.g.G * p.splits);
    if (p.dg) return launch_kernel(conv_fwd_simt_kernel<T, BM, VEC, true>, grid, dim3(THREADS), 0, stream, p.pdl != 0, 1, p);
    return launch_kernel(conv_fwd_simt_kernel<T, BM, VEC, false>, grid, dim3(THREADS), 0, stream, p.pdl != 0, 1, p);
}

}  // namespace

cudaError_t launch_simt(const SimtParams& p, bool bf16, int BM, bool vec, cudaStream_t stream) {
    if (bf16) {
        if (BM == 128) return vec ? launch_t<__nv_bfloat16, 128, true>(p, stream) : launch_t<__nv_bfloat16, 128, false>(p, stream);
        return vec ? launch_t<__nv_bfloat16, 64, true>(p, stream) : launch_t<__nv_bfloat16, 64, false>(p, stream);
    }
    if (BM == 128) return vec ? launch_t<float, 128, true>(p, stream) : launch_t<float, 128, false>(p, stream);
    return vec ? launch_t<float, 64, true>(p, stream) : launch_t<float, 64, false>(p, stream);
}

}  // namespace convfwd
