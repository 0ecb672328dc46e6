// Microbenchmark of the fused scan kernel's consumer loop (4 states per lane,
// 4 lanes per channel, 32-step blocks, bf16 inputs) with the stage data
// resident in shared memory: no TMA ring and no waits, the same helpers and
// arithmetic as scan_kernel.  Prints cycles per step of one warp with 1, 2 and
// 3 consumer warps per SM sub-partition, for the loop as it is, without the
// exponentials, and without the B/C loads (constants instead), to show which
// resource bounds it.  Build and run (one GPU):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 --expt-relaxed-constexpr -I include \
//        -o /tmp/probe_scan_loop selective_state_space_02_gb300/probe_scan_loop.cu && /tmp/probe_scan_loop
#include <cstdio>
#include "csrc/scan_fused_impl.cuh"

using namespace ssm;
using namespace ssm::fused;

constexpr int S = 4, NP = 16, NS = NP / S, CPW = 32 / NS, KB = 32, E = KB / NS, TC = 32;
constexpr int BCW = bc_row(NP, S);
using T = __nv_bfloat16;

template <int VAR>
__global__ void __launch_bounds__(384, 1) probe(int ntiles, float *out) {
    __shared__ __align__(16) float BCs[TC * BCW];
    __shared__ __align__(16) __nv_bfloat16 xs[12 * CPW * TC], ds[12 * CPW * TC], zs[12 * CPW * TC];
    for (int i = threadIdx.x; i < TC * BCW; i += blockDim.x) BCs[i] = 0.01f * (i % 37) - 0.15f;
    for (int i = threadIdx.x; i < 12 * CPW * TC; i += blockDim.x) {
        xs[i] = __float2bfloat16(0.01f * (i % 29) - 0.1f);
        ds[i] = __float2bfloat16(0.05f * (i % 13) - 0.3f);
        zs[i] = __float2bfloat16(0.02f * (i % 17) - 0.2f);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cw = lane / NS, g = lane % NS;
    const int cl = warp * CPW + cw;
    const int own0 = g * E;
    const unsigned char *bx = reinterpret_cast<const unsigned char *>(xs);
    const unsigned char *bd = reinterpret_cast<const unsigned char *>(ds);
    const unsigned char *bz = reinterpret_cast<const unsigned char *>(zs);
    float2 h2[S / 2], a2[S / 2];
    for (int q = 0; q < S / 2; ++q) { a2[q] = make_float2(-1.0f - q - 0.1f * g, -2.0f - q); h2[q] = make_float2(0, 0); }
    const float bias = 0.1f, Dd = 0.5f;
    float check = 0.0f;
    for (int tile = 0; tile < ntiles; ++tile) {
        const float *BC = BCs;
        const int cb = 0, ce = own0;
        float Dl[E], Ul[E], xv[E];
        {
            float dv[E];
            rawE<T, E>(bd, cl * TC + ce, dv);
            rawE<T, E>(bx, cl * TC + ce, xv);
#pragma unroll
            for (int k = 0; k < E; k += 2) {
                const float2 v = __fadd2_rn(make_float2(dv[k], dv[k + 1]), make_float2(bias, bias));
                float2 Dv = softplus2(v);
                const float2 Uv = __fmul2_rn(Dv, make_float2(xv[k], xv[k + 1]));
                Dl[k] = Dv.x; Dl[k + 1] = Dv.y;
                Ul[k] = Uv.x; Ul[k + 1] = Uv.y;
            }
        }
        constexpr int JB = 4;
        float pv[KB];
#pragma unroll
        for (int j0 = 0; j0 < KB; j0 += JB) {
            float2 av[JB][S / 2], bv[JB][S / 2], cv[JB][S / 2];
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                const int j = j0 + jj;
                const int src = (lane & ~(NS - 1)) | (j / E);
                const float Dj = __shfl_sync(0xffffffffu, Dl[j % E], src);
                const float Uj = __shfl_sync(0xffffffffu, Ul[j % E], src);
                const float2 dd = make_float2(Dj, Dj), uu = make_float2(Uj, Uj);
                const float *bc = BC + (cb + j) * BCW + g * bc_group(S);
                float bcv[2 * S];
#pragma unroll
                for (int k = 0; k < 2 * S; k += 4) {
                    const float4 v4 = VAR == 6 ? make_float4(0.01f * k, 0.02f, -0.01f * j, 0.03f) : *reinterpret_cast<const float4 *>(bc + k);
                    bcv[k] = v4.x; bcv[k + 1] = v4.y; bcv[k + 2] = v4.z; bcv[k + 3] = v4.w;
                }
#pragma unroll
                for (int q = 0; q < S / 2; ++q) {
                    const float2 arg = __fmul2_rn(dd, a2[q]);
                    if (VAR == 3) av[jj][q] = __fmul2_rn(arg, make_float2(0.5f, 0.5f));   // multiply instead
                    else av[jj][q] = make_float2(ex2(arg.x), ex2(arg.y));
                    bv[jj][q] = __fmul2_rn(uu, make_float2(bcv[2 * q], bcv[2 * q + 1]));
                    cv[jj][q] = make_float2(bcv[S + 2 * q], bcv[S + 2 * q + 1]);
                }
            }
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
                float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int q = 0; q < S / 2; ++q) {
                    h2[q] = __ffma2_rn(av[jj][q], h2[q], bv[jj][q]);
                    if (q % 2 == 0) acc0 = __ffma2_rn(cv[jj][q], h2[q], acc0);
                    else acc1 = __ffma2_rn(cv[jj][q], h2[q], acc1);
                }
                const float2 acc = __fadd2_rn(acc0, acc1);
                pv[j0 + jj] = acc.x + acc.y;
            }
        }
        ReduceScatter<KB / 2, NS / 2>::run(pv, g);
        float zv[E];
        rawE<T, E>(bz, cl * TC + ce, zv);
#pragma unroll
        for (int k = 0; k < E; k += 2) {
            float2 v = __ffma2_rn(make_float2(Dd, Dd), make_float2(xv[k], xv[k + 1]), make_float2(pv[k], pv[k + 1]));
            v = __fmul2_rn(v, make_float2(gate<T>(zv[k]), gate<T>(zv[k + 1])));
            check += v.x + v.y;
        }
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = check + h2[0].x + h2[1].y;
}


template <int VAR>
void run(const char *name, float *out) {
    for (int wps : {1, 2, 3}) {               // consumer warps per SM sub-partition
        const int warps = 4 * wps;
        const int ntiles = 512;
        probe<VAR><<<152, warps * 32>>>(8, out);
        cudaEvent_t a, b; cudaEventCreate(&a); cudaEventCreate(&b);
        cudaEventRecord(a);
        probe<VAR><<<152, warps * 32>>>(ntiles, out);
        cudaEventRecord(b); cudaEventSynchronize(b);
        float ms = 0; cudaEventElapsedTime(&ms, a, b);
        const double cyc = ms * 1e-3 * 2.07e9 / (ntiles * 32.0);   // at the 2070 MHz maximum SM clock
        printf("%-16s warps/SMSP %d  %7.3f ms  %6.1f cycles/step/warp  %5.1f%% of the 32-updates/clk/SM peak\n",
               name, wps, ms, cyc, 100.0 * warps * 32 * S / cyc / 32.0);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) { printf("error %s\n", cudaGetErrorString(e)); return; }
    }
}

int main() {
    float *out; cudaMalloc(&out, 152 * 384 * 4);
    run<0>("loop", out);
    run<3>("no exponentials", out);
    run<6>("no B/C loads", out);
    cudaFree(out);
    return 0;
}
