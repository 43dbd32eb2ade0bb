// CUDA-core GEMM with fp32 accumulation: the arithmetic of the fp32 layer type (every
// contraction of the layer; the bf16 type uses the tcgen05 kernels instead).
//
// C[r, n] = epilogue( sum_seg sum_k A_seg[arow(r), k] * B_seg[n, k] )
//   arow(r) = a_index ? a_index[r] : r         (row gather, e.g. tokens of one expert)
//   grouped: blockIdx.z = group g, rows [off[g], off[g+1]), B_seg += g * b_group_stride
//   GLU epilogue: the up half of column n reads B row n + glu_up_row and the output is
//   SiTU(gate) * softcap(up) (K3 architecture write-up, SiTU激活优化).
//   SIGMOID epilogue: sigmoid(acc + mu[n]) (the router scores).
#include "common.cuh"
#include "internal.h"

namespace slmoe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

template <typename TA, typename TB, typename TC, int EPI>
__global__ void __launch_bounds__(NT) simt_gemm_kernel(SimtGemm p) {
    const int g = blockIdx.z;
    int row_begin = 0, row_end = p.M;
    if (p.group_offsets) {
        row_begin = p.group_offsets[g];
        row_end = p.group_offsets[g + 1];
    }
    const int m0 = row_begin + blockIdx.y * BM;
    if (m0 >= row_end) return;
    const int n0 = blockIdx.x * BN;

    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    __shared__ float Us[EPI == SIMT_GLU ? BK : 1][BN + 4];
    __shared__ int arow[BM];

    const int tid = threadIdx.x;
    if (tid < BM) {
        int r = m0 + tid;
        arow[tid] = (r < row_end) ? (p.a_index ? p.a_index[r] : r) : -1;
    }
    __syncthreads();

    const int tx = tid % 16, ty = tid / 16;
    float acc[4][4], accu[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = accu[i][j] = 0.f;

    for (int s = 0; s < p.nseg; ++s) {
        const SimtSeg sg = p.seg[s];
        const TA *A = static_cast<const TA *>(sg.A);
        const TB *B = static_cast<const TB *>(sg.B) + (int64_t)g * sg.b_group_stride;
        for (int k0 = 0; k0 < sg.K; k0 += BK) {
            for (int i = tid; i < BM * BK; i += NT) {
                int r = i / BK, kk = i % BK, kg = k0 + kk;
                int ar = arow[r];
                As[kk][r] = (ar >= 0 && kg < sg.K) ? to_f32(A[(int64_t)ar * sg.lda + kg]) : 0.f;
            }
            for (int i = tid; i < BN * BK; i += NT) {
                int c = i / BK, kk = i % BK, kg = k0 + kk, n = n0 + c;
                bool ok = (n < p.N) && (kg < sg.K);
                Bs[kk][c] = ok ? to_f32(B[(int64_t)n * sg.ldb + kg]) : 0.f;
                if (EPI == SIMT_GLU)
                    Us[kk][c] = ok ? to_f32(B[(int64_t)(n + p.glu_up_row) * sg.ldb + kg]) : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                float a[4], b[4], u[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    b[j] = Bs[kk][tx * 4 + j];
                    if (EPI == SIMT_GLU) u[j] = Us[kk][tx * 4 + j];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                        if (EPI == SIMT_GLU) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
                    }
            }
            __syncthreads();
        }
    }

    TC *C = static_cast<TC *>(p.C);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int r = m0 + ty * 4 + i;
        if (r >= row_end) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int n = n0 + tx * 4 + j;
            if (n >= p.N) continue;
            float v = acc[i][j];
            if (EPI == SIMT_GLU) {
                v = situ_glu_accurate(v, accu[i][j], p.beta1, p.beta2);
            } else if (EPI == SIMT_SIGMOID) {
                if (p.mu) v += p.mu[n];
                v = 1.0f / (1.0f + expf(-v));
            }
            C[(int64_t)r * p.ldc + n] = from_f32<TC>(v);
        }
    }
}

template <typename TA, typename TB, typename TC, int EPI>
int run(const SimtGemm &g, cudaStream_t st) {
    dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM, g.groups);
    if (grid.x == 0 || grid.y == 0 || grid.z == 0) return SLMOE_OK;
    if (grid.y > 65535 || grid.z > 65535)
        return fail(SLMOE_EUNSUPPORTED, "simt gemm grid too large (%u, %u)", grid.y, grid.z);
    simt_gemm_kernel<TA, TB, TC, EPI><<<grid, NT, 0, st>>>(g);
    return check_launch("simt_gemm");
}

}  // namespace

int launch_simt_gemm(const SimtGemm &g, cudaStream_t st) {
    using bf = __nv_bfloat16;
    const int key = (g.a_type << 6) | (g.b_type << 5) | (g.c_type << 4) | g.epi;
#define K_(a, b, c, e) (((a) << 6) | ((b) << 5) | ((c) << 4) | (e))
    switch (key) {
    case K_(DT_F32, DT_F32, DT_F32, SIMT_STORE): return run<float, float, float, SIMT_STORE>(g, st);
    case K_(DT_F32, DT_F32, DT_F32, SIMT_GLU): return run<float, float, float, SIMT_GLU>(g, st);
    case K_(DT_F32, DT_F32, DT_F32, SIMT_SIGMOID): return run<float, float, float, SIMT_SIGMOID>(g, st);
    case K_(DT_BF16, DT_F32, DT_F32, SIMT_SIGMOID): return run<bf, float, float, SIMT_SIGMOID>(g, st);
    case K_(DT_BF16, DT_BF16, DT_BF16, SIMT_STORE): return run<bf, bf, bf, SIMT_STORE>(g, st);
    case K_(DT_BF16, DT_BF16, DT_BF16, SIMT_GLU): return run<bf, bf, bf, SIMT_GLU>(g, st);
    default: return fail(SLMOE_EUNSUPPORTED, "simt gemm: no kernel for type key %d", key);
    }
#undef K_
}

}  // namespace slmoe
