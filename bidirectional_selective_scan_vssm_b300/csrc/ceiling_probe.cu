// Throughput ceilings of the two pipes the scan's recurrence runs on, measured
// on the GPU it runs on: the MUFU exp2 unit (ex2.approx.ftz.f32) and the fp32
// FMA pipe (scalar and packed f32x2), alone and mixed at the recurrence's
// ratio of one exp to four fp32 operations. Prints one JSON line.
//
//     python bidirectional_selective_scan_vssm_b300/build.py --probe
//     bidirectional_selective_scan_vssm_b300/ceiling_probe
//
// Each thread runs independent register-only chains; every result is written
// out so that nothing is optimised away.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include "ptx.cuh"

namespace {

constexpr int kIters = 2048;
constexpr int kChains = 8;

__global__ void mufu_ex2(float *out, float s)
{
    float v[kChains];
    for (int i = 0; i < kChains; ++i) v[i] = s * (threadIdx.x + i) * 1e-4f;
    for (int it = 0; it < kIters; ++it)
#pragma unroll
        for (int i = 0; i < kChains; ++i) v[i] = vssm::ex2_mufu(-v[i]);   // stays in (0.5, 1]
    float a = 0.f;
    for (int i = 0; i < kChains; ++i) a += v[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = a;
}

__global__ void fma_scalar(float *out, float s)
{
    float v[kChains];
    for (int i = 0; i < kChains; ++i) v[i] = s * (threadIdx.x + i);
    const float b = 0.999f, c = 1e-3f * s;
    for (int it = 0; it < kIters; ++it)
#pragma unroll
        for (int i = 0; i < kChains; ++i) v[i] = fmaf(v[i], b, c);
    float a = 0.f;
    for (int i = 0; i < kChains; ++i) a += v[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = a;
}

__global__ void fma_packed(float *out, float s)
{
    vssm::f2 v[kChains];
    for (int i = 0; i < kChains; ++i) v[i] = vssm::pack2(s + i, 0.5f * s + threadIdx.x);
    const vssm::f2 b = vssm::pack2(0.999f, 0.998f), c = vssm::pack2(1e-3f * s, 2e-3f);
    for (int it = 0; it < kIters; ++it)
#pragma unroll
        for (int i = 0; i < kChains; ++i) v[i] = vssm::fma2(v[i], b, c);
    float a = 0.f;
    for (int i = 0; i < kChains; ++i) {
        const float2 q = vssm::unpack2(v[i]);
        a += q.x + q.y;
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = a;
}

// One exp2 per four fp32 operations (two packed FMAs), as in the recurrence.
__global__ void mixed(float *out, float s)
{
    float v[kChains];
    vssm::f2 w[kChains];
    for (int i = 0; i < kChains; ++i) {
        v[i] = s * (threadIdx.x + i) * 1e-4f;
        w[i] = vssm::pack2(s + i, 0.5f * s);
    }
    const vssm::f2 b = vssm::pack2(0.999f, 0.998f), c = vssm::pack2(1e-3f * s, 2e-3f);
    for (int it = 0; it < kIters; ++it)
#pragma unroll
        for (int i = 0; i < kChains; ++i) {
            v[i] = vssm::ex2_mufu(-v[i]);
            w[i] = vssm::fma2(vssm::fma2(w[i], b, c), b, c);
        }
    float a = 0.f;
    for (int i = 0; i < kChains; ++i) {
        const float2 q = vssm::unpack2(w[i]);
        a += v[i] + q.x + q.y;
    }
    out[blockIdx.x * blockDim.x + threadIdx.x] = a;
}

// Per-SM-per-clock rate of `ops_per_thread_iter` operations.
double rate(void (*k)(float *, float), float *out, int blocks, int threads, double ops_per_thread_iter,
            double sm_clock_hz, int sms)
{
    for (int r = 0; r < 3; ++r) k<<<blocks, threads>>>(out, 1.0f);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a);
    const int reps = 10;
    for (int r = 0; r < reps; ++r) k<<<blocks, threads>>>(out, 1.0f);
    cudaEventRecord(b);
    cudaEventSynchronize(b);
    float ms = 0.f;
    cudaEventElapsedTime(&ms, a, b);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    const double ops = (double)reps * blocks * threads * kIters * ops_per_thread_iter;
    return ops / (ms * 1e-3) / sms / sm_clock_hz;
}

}  // namespace

int main()
{
    int sms = 0, khz = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, 0);
    const int blocks = sms * 4, threads = 512;
    float *out = nullptr;
    if (cudaMalloc(&out, sizeof(float) * blocks * threads) != cudaSuccess) {
        printf("{\"error\": \"cudaMalloc failed\"}\n");
        return 1;
    }
    const double hz = khz * 1e3;   // rates below are per clock at the maximum SM clock
    const double ex2 = rate(mufu_ex2, out, blocks, threads, kChains, hz, sms);
    const double ffma = rate(fma_scalar, out, blocks, threads, kChains, hz, sms);
    const double ffma2 = rate(fma_packed, out, blocks, threads, 2.0 * kChains, hz, sms);
    const double mix = rate(mixed, out, blocks, threads, kChains, hz, sms);
    const cudaError_t e = cudaGetLastError();
    cudaFree(out);
    printf("{\"sms\": %d, \"max_sm_mhz\": %.0f, \"ex2_per_clk_sm\": %.2f, \"ffma_lane_ops_per_clk_sm\": %.2f, "
           "\"ffma2_lane_ops_per_clk_sm\": %.2f, \"mixed_ex2_per_clk_sm\": %.2f, \"status\": \"%s\"}\n",
           sms, khz / 1e3, ex2, ffma, ffma2, mix, cudaGetErrorString(e));
    return e == cudaSuccess ? 0 : 1;
}
