// Weighted top-k combine at the source: out[t] = sum_j gate[t, j] * Ret[ret_slot[t, j]], fp32,
// j ascending. "Fine-grained Computation-Communication Overlap via Tile-level Signaling and
// Scheduling for Mixture-of-Experts" (pith.science/paper/W2ZARMHG), "Axiom & Free-Parameter
// Ledger": the combine plan (ret_slot) is resolved before the return path runs.
#include "moe_internal.cuh"

namespace moe {

constexpr int KMAX_C = 8;

// One warp per token; each lane handles 8 consecutive columns per step (16-byte bf16 loads,
// two 16-byte fp32 stores).
__global__ void __launch_bounds__(256) combine_kernel(Shape s, PlanPtrs p, float* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int vec = s.d / 8;
    const uint4* ret = reinterpret_cast<const uint4*>(p.Ret);
    const int rows = s.T * s.k;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < s.T; t += nwarps) {
        int my_slot = 0;
        float my_w = 0.f;
        if (lane < s.k) {
            my_slot = p.ret_slot[(size_t)t * s.k + lane];
            my_w = p.gate[(size_t)t * s.k + lane];
        }
        int sl[KMAX_C];
        float w[KMAX_C];
        bool good = true;
#pragma unroll
        for (int j = 0; j < KMAX_C; ++j) {
            sl[j] = __shfl_sync(0xffffffffu, my_slot, j);
            w[j] = __shfl_sync(0xffffffffu, my_w, j);
            if (j < s.k) good &= (sl[j] >= 0 && sl[j] < rows);
        }
        if (!good) {
            if (lane == 0) set_status(p.meta, ST_BAD_PLAN, t);
            continue;
        }
        float4* o = reinterpret_cast<float4*>(out + (size_t)t * s.d);
        for (int v = lane; v < vec; v += 32) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < KMAX_C; ++j) {
                if (j >= s.k) break;
                const uint4 r = ret[(size_t)sl[j] * vec + v];
                const uint32_t q[4] = {r.x, r.y, r.z, r.w};
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
    combine_kernel<<<blocks, 256, 0, st>>>(s, p, out);
    return cudaGetLastError();
}

}  // namespace moe
