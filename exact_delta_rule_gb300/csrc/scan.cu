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
constexpr int KT = 32;   // columns of M staged per step

__global__ void __launch_bounds__(256) scan_combine_kernel(const float *__restrict__ S0, const float *__restrict__ maps,
                                                           float *__restrict__ s_in, int B, int G, int H) {
    __shared__ float cur[D][CB];          // S_in[g-1][:, cols]
    __shared__ float mt[D][KT + 1];       // a K-slice of M_{g-1}
    const int tid = threadIdx.x;
    const int cb = blockIdx.x % (D / CB);
    const int bh = blockIdx.x / (D / CB);
    const int b = bh / H, h = bh % H;
    const int c0 = cb * CB;
    const size_t mat = (size_t)D * D;
    // S_in[0] = S0 (or zero)
    for (int e = tid; e < D * CB; e += 256) {
        const int r = e / CB, c = e % CB;
        const float x = S0 ? S0[((size_t)b * H + h) * mat + (size_t)r * D + c0 + c] : 0.f;
        cur[r][c] = x;
        s_in[(((size_t)b * G + 0) * H + h) * mat + (size_t)r * D + c0 + c] = x;
    }
    __syncthreads();
    const int r = tid >> 1, ch = (tid & 1) * 8;  // this thread's row and 8 of the block's columns
    for (int g = 1; g < G; ++g) {
        const float *M = maps + (((size_t)0 * B + b) * (G - 1) + (g - 1)) * H * mat + (size_t)h * mat;
        const float *N = maps + (((size_t)1 * B + b) * (G - 1) + (g - 1)) * H * mat + (size_t)h * mat;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = N[(size_t)r * D + c0 + ch + j];
        for (int k0 = 0; k0 < D; k0 += KT) {
            for (int e = tid; e < D * KT; e += 256) {  // rows of M are contiguous: coalesced along k
                const int rr = e / KT, kk = e % KT;
                mt[rr][kk] = M[(size_t)rr * D + k0 + kk];
            }
            __syncthreads();
#pragma unroll 4
            for (int kk = 0; kk < KT; ++kk) {
                const float m = mt[r][kk];
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(m, cur[k0 + kk][ch + j], acc[j]);
            }
            __syncthreads();
        }
        // every thread has read cur for this step (barrier above): overwrite it
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            cur[r][ch + j] = acc[j];
            s_in[(((size_t)b * G + g) * H + h) * mat + (size_t)r * D + c0 + ch + j] = acc[j];
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_scan_combine(const float *S0, const float *maps, float *s_in, int B, int G, int H,
                                cudaStream_t stream) {
    if (B == 0 || G == 0) return cudaSuccess;
    scan_combine_kernel<<<(unsigned)(B * H * (D / CB)), 256, 0, stream>>>(S0, maps, s_in, B, G, H);
    return cudaGetLastError();
}

}  // namespace efla
