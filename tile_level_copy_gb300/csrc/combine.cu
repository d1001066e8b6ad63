// Weighted top-k combine at the source: out[t] = sum_j gate[t, j] * Ret[ret_slot[t, j]], fp32,
// j ascending. "Fine-grained Computation-Communication Overlap via Tile-level Signaling and
// Scheduling for Mixture-of-Experts" (pith.science/paper/W2ZARMHG), "Axiom & Free-Parameter
// Ledger": the combine plan (ret_slot) is resolved before the return path runs.
#include "moe_internal.cuh"

namespace moe {

// One warp per token; each lane handles 8 consecutive columns per step (16-byte bf16 loads,
// two 16-byte fp32 stores). The k rows' loads of a step are all issued before any is used (and the
// next token's slots and gates are fetched while the current token is combined), so each lane has
// k loads in flight instead of one.
template <int K>  // K = top-k, so that the per-lane arrays have exactly K entries
__global__ void __launch_bounds__(256, 4) combine_kernel(Shape s, PlanPtrs p, float* __restrict__ out) {
    griddep_wait();  // the return copy (and every row of Ret) is complete
    griddep_launch();  // MOE_PDL: the next layer's routing kernel may start; it waits for this grid
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int vec = s.d / 8;
    constexpr int k = K;
    const uint4* ret = reinterpret_cast<const uint4*>(p.Ret);
    const int rows = s.T * k;
    int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int nx_slot = 0;
    float nx_w = 0.f;
    if (t < s.T && lane < k) {
        nx_slot = __ldg(p.ret_slot + (size_t)t * k + lane);
        nx_w = __ldg(p.gate + (size_t)t * k + lane);
    }
    for (; t < s.T; t += nwarps) {
        const int my_slot = nx_slot;
        const float my_w = nx_w;
        const int tn = t + nwarps;
        if (tn < s.T && lane < k) {  // the next token's plan entries, in flight meanwhile
            nx_slot = __ldg(p.ret_slot + (size_t)tn * k + lane);
            nx_w = __ldg(p.gate + (size_t)tn * k + lane);
        }
        int sl[K];
        float w[K];
        bool good = true;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            sl[j] = __shfl_sync(0xffffffffu, my_slot, j);
            w[j] = __shfl_sync(0xffffffffu, my_w, j);
            good &= (sl[j] >= 0 && sl[j] < rows);
        }
        if (!good) {
            if (lane == 0) set_status(p.meta, ST_BAD_PLAN, t);
            continue;
        }
        float4* o = reinterpret_cast<float4*>(out + (size_t)t * s.d);
        for (int v = lane; v < vec; v += 32) {
            uint4 r[K];
#pragma unroll
            for (int j = 0; j < K; ++j) r[j] = ret[(size_t)sl[j] * vec + v];
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const uint32_t q[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = __uint_as_float(q[i] << 16);
                    const float hi = __uint_as_float(q[i] & 0xffff0000u);
                    acc[2 * i] = fmaf(w[j], lo, acc[2 * i]);
                    acc[2 * i + 1] = fmaf(w[j], hi, acc[2 * i + 1]);
                }
            }
            o[2 * v] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            o[2 * v + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
}

cudaError_t launch_combine(const Shape& s, const PlanPtrs& p, float* out, int sms, cudaStream_t st) {
    const int blocks = min((s.T + 7) / 8, sms * 8);
    const bool pdl = (s.flags & MOE_PDL) != 0;
    const dim3 g(blocks), b(256);
    switch (s.k) {
        case 1: return launch_k(combine_kernel<1>, g, b, 0, st, pdl, s, p, out);
        case 2: return launch_k(combine_kernel<2>, g, b, 0, st, pdl, s, p, out);
        case 3: return launch_k(combine_kernel<3>, g, b, 0, st, pdl, s, p, out);
        case 4: return launch_k(combine_kernel<4>, g, b, 0, st, pdl, s, p, out);
        case 5: return launch_k(combine_kernel<5>, g, b, 0, st, pdl, s, p, out);
        case 6: return launch_k(combine_kernel<6>, g, b, 0, st, pdl, s, p, out);
        case 7: return launch_k(combine_kernel<7>, g, b, 0, st, pdl, s, p, out);
        case 8: return launch_k(combine_kernel<8>, g, b, 0, st, pdl, s, p, out);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
