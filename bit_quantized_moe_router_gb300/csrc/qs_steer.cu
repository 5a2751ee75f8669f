// qs_steer.cu -- directional steering of the layer's output rows (sm_103a).
//
// Every token row y of the FFN output is edited in place as
//     y <- y - scale * d * (d . y)
// (QuarkStar (q36) README, "Steering"; the DwarfStar (ds4) page's "Steering"
// section uses the same projection), d being the layer's direction as given.
//
// One CTA per token row.  A thread owns every 256th group of four elements: it
// reads them once for the dot product (the row then sits in L1 for the second
// pass), the eight warp sums are added in a fixed order, so the result does not
// depend on scheduling, and the same thread rewrites its groups.  The row is
// read twice from the SM's point of view and once from HBM; HBM traffic per
// call is T*H*4 bytes in, T*H*4 out and H*4 for the direction.
//
// The kernel is a programmatic dependent launch: it may start while the kernel
// before it in the stream (the layer) still runs, loads its share of the
// direction (a parameter, never written by that kernel), and waits for that
// kernel's grid to finish (griddepcontrol.wait) before it reads a row.  It lets
// the kernel after it launch as soon as every CTA of it has started.
#include "qs_common.cuh"
#include "qs_internal.h"

namespace qs {

constexpr int kSteerThreads = 256;

__global__ void __launch_bounds__(kSteerThreads) steer_rows_kernel(float* __restrict__ y, const float* __restrict__ d,
                                                                   float scale, int H) {
    __shared__ float part[kSteerThreads / 32];
    float4* row = reinterpret_cast<float4*>(y + (size_t)blockIdx.x * H);
    const float4* dir = reinterpret_cast<const float4*>(d);
    const int n4 = H >> 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the first two groups of the direction this thread uses (all of it for H <= 2048)
    const int i0 = threadIdx.x, i1 = threadIdx.x + kSteerThreads;
    const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float4 d0 = i0 < n4 ? __ldg(dir + i0) : z4, d1 = i1 < n4 ? __ldg(dir + i1) : z4;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    auto dir_at = [&](int i) { return i == i0 ? d0 : (i == i1 ? d1 : __ldg(dir + i)); };
    float acc = 0.0f;
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += kSteerThreads) {
        const float4 a = row[i], b = dir_at(i);
        acc = fmaf(a.x, b.x, acc);
        acc = fmaf(a.y, b.y, acc);
        acc = fmaf(a.z, b.z, acc);
        acc = fmaf(a.w, b.w, acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) part[warp] = acc;
    __syncthreads();
    float c = 0.0f;
#pragma unroll
    for (int w = 0; w < kSteerThreads / 32; w++) c += part[w];
    const float f = scale * c;
#pragma unroll 4
    for (int i = threadIdx.x; i < n4; i += kSteerThreads) {
        float4 a = row[i];
        const float4 b = dir_at(i);
        a.x = fmaf(-f, b.x, a.x);
        a.y = fmaf(-f, b.y, a.y);
        a.z = fmaf(-f, b.z, a.z);
        a.w = fmaf(-f, b.w, a.w);
        row[i] = a;
    }
}

cudaError_t launch_steer_rows(float* y, const float* d, float scale, int T, int H, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T);
    cfg.blockDim = dim3(kSteerThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, steer_rows_kernel, y, d, scale, H);
}

}  // namespace qs
