// Start states of the segments of a split sequence.
//
// Over any stretch of tokens the recurrence S <- (I - alpha k k^T) S + alpha k v^T
// ["Exact Flow Linear Attention" (gist.science), Metodologia 3] is affine in its
// start state: S_out = M S_in + N, with M the product of the stretch's factors
// (I - alpha_t k_t k_t^T) (the stretch run from S = I with v = 0) and N the
// stretch run from S = 0.  With the maps (M_g, N_g) of segments g = 0..G-2 of a
// sequence, the start state of segment g is
//   S_in[0] = S0,   S_in[g] = M_{g-1} S_in[g-1] + N_{g-1},
// a short serial scan of d_k x d_k by d_k x d_v products.  The columns of S are
// independent, so one CTA handles a block of 16 columns of one (b, h) through
// all G segments, in fp32 on CUDA cores.
#include "internal.cuh"

namespace efla {
namespace {

constexpr int D = 128;
constexpr int CB = 16;   // columns of S per CTA
constexpr int MLD = D + 4;  // row stride of a staged map (16-byte aligned rows)
constexpr size_t DYN_SMEM = 2 * (size_t)D * MLD * sizeof(float);  // two maps in flight

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__global__ void __launch_bounds__(256) scan_combine_kernel(const float *__restrict__ S0, const float *__restrict__ maps,
                                                           float *__restrict__ s_in, int B, int G, int H) {
    extern __shared__ __align__(16) float mbuf[];  // [2][D][MLD]: M_{g-1}, then M_g while step g runs
    __shared__ __align__(16) float cur[D][CB];     // S_in[g-1][:, cols]
    const int tid = threadIdx.x;
    const int cb = blockIdx.x % (D / CB);
    const int bh = blockIdx.x / (D / CB);
    const int b = bh / H, h = bh % H;
    const int c0 = cb * CB;
    const size_t mat = (size_t)D * D;
    auto Mptr = [&](int g) { return maps + (((size_t)0 * B + b) * (G - 1) + g) * H * mat + (size_t)h * mat; };
    auto Nptr = [&](int g) { return maps + (((size_t)1 * B + b) * (G - 1) + g) * H * mat + (size_t)h * mat; };
    auto fetch_M = [&](int g, int buf) {  // 64 KB, 16 bytes per copy, 16 copies per thread
        const float *M = Mptr(g);
        float *dst = mbuf + (size_t)buf * D * MLD;
#pragma unroll
        for (int x = 0; x < D * D / 4 / 256; ++x) {
            const int e = tid + x * 256, r = e / (D / 4), c4 = e % (D / 4);
            cp_async16(dst + r * MLD + 4 * c4, M + (size_t)r * D + 4 * c4);
        }
        cp_async_commit();
    };
    if (G > 1) fetch_M(0, 0);
    // S_in[0] = S0 (or zero)
    for (int e = tid; e < D * CB; e += 256) {
        const int r = e / CB, c = e % CB;
        const float x = S0 ? S0[((size_t)b * H + h) * mat + (size_t)r * D + c0 + c] : 0.f;
        cur[r][c] = x;
        s_in[(((size_t)b * G + 0) * H + h) * mat + (size_t)r * D + c0 + c] = x;
    }
    const int r = tid >> 1, ch = (tid & 1) * 8;  // this thread's row and 8 of the block's columns
    for (int g = 1; g < G; ++g) {
        const int buf = (g - 1) & 1;
        float acc[8];
        const float *N = Nptr(g - 1);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = N[(size_t)r * D + c0 + ch + j];
        if (g + 1 < G) {  // the next map streams in while this step runs
            fetch_M(g, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // M_{g-1} and S_in[g-1] visible to every thread
        const float *Mr = mbuf + (size_t)buf * D * MLD + (size_t)r * MLD;
#pragma unroll 4
        for (int k = 0; k < D; k += 4) {
            const float4 m4 = *reinterpret_cast<const float4 *>(Mr + k);
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 a = *reinterpret_cast<const float4 *>(&cur[k + e][ch]);
                const float4 c = *reinterpret_cast<const float4 *>(&cur[k + e][ch + 4]);
                acc[0] = fmaf(mv[e], a.x, acc[0]);
                acc[1] = fmaf(mv[e], a.y, acc[1]);
                acc[2] = fmaf(mv[e], a.z, acc[2]);
                acc[3] = fmaf(mv[e], a.w, acc[3]);
                acc[4] = fmaf(mv[e], c.x, acc[4]);
                acc[5] = fmaf(mv[e], c.y, acc[5]);
                acc[6] = fmaf(mv[e], c.z, acc[6]);
                acc[7] = fmaf(mv[e], c.w, acc[7]);
            }
        }
        __syncthreads();  // every thread has read cur and this map buffer
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            cur[r][ch + j] = acc[j];
            s_in[(((size_t)b * G + g) * H + h) * mat + (size_t)r * D + c0 + ch + j] = acc[j];
        }
    }
}

}  // namespace

cudaError_t launch_scan_combine(const float *S0, const float *maps, float *s_in, int B, int G, int H,
                                cudaStream_t stream) {
    if (B == 0 || G == 0) return cudaSuccess;
    static bool attr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64 || !attr[dev]) {
        e = cudaFuncSetAttribute(scan_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DYN_SMEM);
        if (e != cudaSuccess) return e;
        if (dev < 64) attr[dev] = true;
    }
    scan_combine_kernel<<<(unsigned)(B * H * (D / CB)), 256, DYN_SMEM, stream>>>(S0, maps, s_in, B, G, H);
    return cudaGetLastError();
}

}  // namespace efla
