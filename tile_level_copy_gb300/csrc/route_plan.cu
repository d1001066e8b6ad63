// Router top-k, per-chunk ranking, the layout plan (histogram, padded offsets, tile-owner map,
// remote-first schedule, segments, return plan, expert-compact rows of the GEMM inputs) and the
// permute of the tokens into those rows.
//
// Method: "Fine-grained Computation-Communication Overlap via Tile-level Signaling and Scheduling
// for Mixture-of-Experts" (pith.science/paper/W2ZARMHG), section "What carries the argument": rows
// of each expert are grouped by owner and every group is padded to a multiple of the tile height so
// that each output tile has one owner; tiles bound for owners are scheduled largest first.
#include "moe_internal.cuh"

namespace moe {

constexpr int ROUTE_THREADS = 256;   // threads per chunk of <= 128 tokens: 2 or more per token
constexpr int KMAX = 8;

// ---------------------------------------------------------------------------------------------
// route_kernel<K>: one CTA per chunk of C = `chunk_tokens` consecutive tokens (a chunk never
// straddles two owners), K = top-k. The chunk's logits are staged in shared memory (16-byte loads
// when the rows allow, rows padded to E+1 words against bank conflicts). TPT = ROUTE_THREADS / C
// threads share a token: each scans every TPT-th logit of the row, keeping a sorted list of its K
// best (value descending, ties to the lower expert id: a logit enters only if strictly greater
// than the list's last, and is inserted after every entry not smaller than it); the TPT lists are
// merged with shuffles, K times taking the best head (value, then lower id) of the group, which is
// the order a single scan of the row gives. The token's first thread forms the gates = softmax over
// the K chosen logits in fp32. Last, thread t of the chunk's first C threads takes token t: each
// warp ORs its lanes into a per-expert lane mask in shared memory, which gives each token's rank
// among the chunk's tokens routed to that expert (ascending token order) and the chunk's count per
// expert.
// ---------------------------------------------------------------------------------------------
template <int K>
__global__ void __launch_bounds__(ROUTE_THREADS) route_kernel(Shape s, const float* __restrict__ logits, PlanPtrs p) {
    extern __shared__ float s_logit[];  // [C][E + 1], then the chosen experts [C][K] (ints)
    __shared__ uint32_t s_mask[ROUTE_THREADS / 32][MAX_E];
    __shared__ int32_t s_wpre[ROUTE_THREADS / 32][MAX_E];

    griddep_launch();  // the plan kernel may start (it waits for this grid before reading)
    // The routing, plan and permute kernels are always launched with programmatic dependent launch
    // (MOE_PDL extends it to the GEMMs and the combine): the kernel before this one on the stream
    // (the caller's, which may have written the logits, or the previous layer's combine, which reads
    // what this grid writes) is complete past this wait
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int C = s.chunk_tokens, E = s.E, ld = E + 1;
    int* s_te = reinterpret_cast<int*>(s_logit + C * ld);
    const int t0 = blockIdx.x * C;
    const float* src = logits + (size_t)t0 * E;
    const int n = C * E;
    if ((E & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        // 16-byte loads, all in flight together (a row is a whole number of vectors)
        const float4* src4 = reinterpret_cast<const float4*>(src);
        const int n4 = n >> 2;
        for (int i0 = tid; i0 < n4; i0 += ROUTE_THREADS * 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * ROUTE_THREADS;
                if (i < n4) v[u] = __ldg(src4 + i);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * ROUTE_THREADS;
                if (i < n4) {
                    float* d = s_logit + ((4 * i) / E) * ld + (4 * i) % E;
                    d[0] = v[u].x;
                    d[1] = v[u].y;
                    d[2] = v[u].z;
                    d[3] = v[u].w;
                }
            }
        }
    } else {
        for (int i0 = tid; i0 < n; i0 += ROUTE_THREADS * 8) {  // eight loads in flight per thread
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * ROUTE_THREADS;
                v[u] = (i < n) ? __ldg(src + i) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * ROUTE_THREADS;
                if (i < n) s_logit[(i / E) * ld + (i % E)] = v[u];
            }
        }
    }
    __syncthreads();
    for (int e = lane; e < E; e += 32) s_mask[warp][e] = 0u;

    // top-K of token tl by its TPT threads (TPT a power of two <= 32, so a token's threads share a
    // warp); threads past the chunk's tokens keep empty lists
    const int TPT = min(ROUTE_THREADS / C, 32), tl = tid / TPT, sub = tid % TPT;
    const bool tok = tl < C;
    {
        const float* row = s_logit + (tok ? tl : 0) * ld;
        float tv[K];
        int te[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            tv[j] = -INFINITY;
            te[j] = -1;
        }
        for (int e = sub; tok && e < E; e += TPT) {
            const float v = row[e];
            if (te[K - 1] < 0 || v > tv[K - 1]) {
                float cv = v;
                int ce = e;
                bool shift = false;  // from the insertion point on, every entry moves down one place
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (shift || te[j] < 0 || cv > tv[j]) {
                        const float fv = tv[j];
                        const int fe = te[j];
                        tv[j] = cv;
                        te[j] = ce;
                        cv = fv;
                        ce = fe;
                        shift = true;
                    }
                }
            }
        }
        // merge: K times, the group's best head (greater value, then lower id; an empty list's head
        // loses) is taken and its list advances
        float mv[K];
        int me[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            float bv = tv[0];
            int be = te[0];
            for (int o = 1; o < TPT; o <<= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                const bool take = oe >= 0 && (be < 0 || ov > bv || (ov == bv && oe < be));
                bv = take ? ov : bv;
                be = take ? oe : be;
            }
            mv[j] = bv;
            me[j] = be;
            if (te[0] == be && be >= 0) {  // this thread's head was taken: pop it
#pragma unroll
                for (int q = 0; q + 1 < K; ++q) {
                    tv[q] = tv[q + 1];
                    te[q] = te[q + 1];
                }
                tv[K - 1] = -INFINITY;
                te[K - 1] = -1;
            }
        }
        if (sub == 0 && tok) {
            float z[K], sum = 0.f;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                z[j] = expf(mv[j] - mv[0]);
                sum += z[j];
            }
            const int t = t0 + tl;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                p.idx[(size_t)t * K + j] = me[j];
                p.gate[(size_t)t * K + j] = z[j] / sum;
                s_te[tl * K + j] = me[j];
            }
        }
    }
    __syncthreads();

    // ranks and counts: thread tid < C takes token tid
    const bool live = tid < C;
    if (live) {
#pragma unroll
        for (int j = 0; j < K; ++j) atomicOr(&s_mask[warp][s_te[tid * K + j]], 1u << lane);
    }
    __syncthreads();
    for (int e = tid; e < E; e += ROUTE_THREADS) {
        int acc = 0;
        for (int w = 0; w < ROUTE_THREADS / 32; ++w) {
            s_wpre[w][e] = acc;
            acc += __popc(s_mask[w][e]);
        }
        p.chunk_cnt[(size_t)blockIdx.x * E + e] = acc;
    }
    __syncthreads();
    if (live) {
        const uint32_t lt = (1u << lane) - 1u;
        const int t = t0 + tid;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int e = s_te[tid * K + j];
            p.rank[(size_t)t * K + j] = s_wpre[warp][e] + __popc(s_mask[warp][e] & lt);
        }
    }
}

template <int K>
static cudaError_t launch_route_k(const Shape& s, const float* logits, const PlanPtrs& p, size_t smem, cudaStream_t st) {
    // the staged logits and chosen experts can take the dynamic shared memory past 48 KB with the
    // static per-warp masks: allow what this launch needs
    const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&route_kernel<K>),
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(route_kernel<K>, dim3(s.n_chunks), dim3(ROUTE_THREADS), smem, st, true, s, logits, p);
}

cudaError_t launch_route(const Shape& s, const float* logits, const PlanPtrs& p, cudaStream_t st) {
    const size_t smem = (size_t)s.chunk_tokens * ((s.E + 1) * sizeof(float) + s.k * sizeof(int));
    switch (s.k) {
        case 1: return launch_route_k<1>(s, logits, p, smem, st);
        case 2: return launch_route_k<2>(s, logits, p, smem, st);
        case 3: return launch_route_k<3>(s, logits, p, smem, st);
        case 4: return launch_route_k<4>(s, logits, p, smem, st);
        case 5: return launch_route_k<5>(s, logits, p, smem, st);
        case 6: return launch_route_k<6>(s, logits, p, smem, st);
        case 7: return launch_route_k<7>(s, logits, p, smem, st);
        case 8: return launch_route_k<8>(s, logits, p, smem, st);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------------------------
// plan_kernel: one CTA of 1024 threads builds the whole plan from the per-chunk counts.
// ---------------------------------------------------------------------------------------------
constexpr int PLAN_THREADS = 1024;
constexpr int PLAN_SMEM_TILES = 16384;  // tiles whose hand-out order and group fit in shared memory (128 KB)

__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* s_total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < PLAN_THREADS / 32) ? s_warp[lane] : 0;
        int wx = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wx, o);
            if (lane >= o) wx += y;
        }
        s_warp[lane] = wx - w;
        if (lane == 31) *s_total = wx;
    }
    __syncthreads();
    const int r = s_warp[warp] + x - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(PLAN_THREADS) plan_kernel(Shape s, PlanPtrs p) {
    griddep_wait();  // the routing kernel's counts
    // The call's status word and layout word are cleared before the permute may start (it runs
    // beside the rest of this kernel once the layout is published, step 5a).
    if (threadIdx.x == 0) {
        p.meta[META_STATUS] = 0;
        p.meta[META_STATUS_DETAIL] = 0;
        p.meta[META_LAYOUT] = 0;
        __threadfence();
    }
    __syncthreads();
    griddep_launch();
    __shared__ int s_n[1024];        // n_{e,r}, group g = e*R + r
    __shared__ int s_off[1025];
    __shared__ int s_load[MAX_E];    // rows per expert
    __shared__ int s_erank[MAX_E];   // position of the expert in (load desc, id asc) order
    __shared__ int s_fb[MAX_E];      // full bands per expert
    __shared__ int s_mt[MAX_E];      // M-tiles per expert
    __shared__ int s_ebase[MAX_E];   // first hand-out position of the expert's bands
    __shared__ int s_cbase[MAX_E];   // first row of the expert in the compact layout
    __shared__ int s_fbp[1024];      // full bands of the groups before g (layout order)
    __shared__ int s_prank[1024];    // rank of group g's partial band among the partial bands
    __shared__ int s_warp[32];
    __shared__ int s_total;

    const int E = s.E, R = s.R, G = E * R, tbM = s.tbM, tid = threadIdx.x;
    const int cpo = (s.T / R) / s.chunk_tokens;  // chunks per owner
    const int slice = (s.T / R) * s.k;           // rows per owner slice of Ret

    // Shared-memory copies of the hand-out order and of each tile's group, read by steps 6 and 7
    // (global memory when the tile count exceeds PLAN_SMEM_TILES).
    extern __shared__ int s_dyn[];
    const bool mirror = s.MT_max <= PLAN_SMEM_TILES;
    int* s_order = s_dyn;
    int* s_tg = s_dyn + (mirror ? s.MT_max : 0);

    // 1. per group: chunk bases (exclusive prefix over the owner's chunks) and n_{e,r}; the counts
    // are read eight at a time so that their loads are in flight together, and neighbouring threads
    // take neighbouring experts of one owner, so that a warp's loads of one chunk are contiguous
    for (int q = tid; q < G; q += PLAN_THREADS) {
        const int r = q / E, e = q % E, g = e * R + r;
        const int32_t* __restrict__ cnt = p.chunk_cnt + e;
        int32_t* __restrict__ base = p.chunk_base + e;
        int acc = 0;
        int c = r * cpo;
        const int c_end = (r + 1) * cpo;
        for (; c + 8 <= c_end; c += 8) {
            int v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __ldcg(cnt + (size_t)(c + i) * E);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                base[(size_t)(c + i) * E] = acc;
                acc += v[i];
            }
        }
        for (; c < c_end; ++c) {
            const int v = __ldcg(cnt + (size_t)c * E);
            base[(size_t)c * E] = acc;
            acc += v;
        }
        s_n[g] = acc;
        p.counts[g] = acc;
    }
    __syncthreads();

    // 2. padded offsets: exclusive scan of ceil(n / tbM) * tbM over g (e-major, r-minor)
    {
        const int g = tid;
        const int padded = (g < G) ? ((s_n[g] + tbM - 1) / tbM) * tbM : 0;
        const int o = block_exclusive_scan(padded, s_warp, &s_total);
        if (g < G) s_off[g] = o;
        if (g == 0) s_off[G] = s_total;
    }
    __syncthreads();
    const int P = s_off[G];
    const int MT = P / tbM;
    for (int g = tid; g <= G; g += PLAN_THREADS) p.offsets[g] = s_off[g];

    // 3. owner return offsets: ret_off[r][e] = sum_{e' < e} n_{e',r}
    for (int r = tid; r < R; r += PLAN_THREADS) {
        int acc = 0;
        for (int e = 0; e < E; ++e) {
            p.ret_off[r * (E + 1) + e] = acc;
            acc += s_n[e * R + r];
        }
        p.ret_off[r * (E + 1) + E] = acc;
    }

    // 4. expert loads, full bands, expert table
    for (int e = tid; e < E; e += PLAN_THREADS) {
        int load = 0, fb = 0;
        for (int r = 0; r < R; ++r) {
            load += s_n[e * R + r];
            fb += s_n[e * R + r] / tbM;
        }
        s_load[e] = load;
        s_fb[e] = fb;
        s_mt[e] = (s_off[(e + 1) * R] - s_off[e * R]) / tbM;
        p.experts[8 * e + 0] = s_off[e * R] / tbM;
        p.experts[8 * e + 1] = s_mt[e];
    }
    __syncthreads();

    // 4b. expert-compact layout of the GEMM inputs: each expert's rows contiguous, the run padded to
    // a multiple of the UMMA tile height BM; inside the run the expert's bands follow one another in
    // hand-out order, each band's valid rows in row order (step 5a places them).
    {
        const int e = tid;
        const int rows = (e < E) ? ((s_load[e] + BM - 1) / BM) * BM : 0;
        const int o = block_exclusive_scan(rows, s_warp, &s_total);
        if (e < E) s_cbase[e] = o;
    }
    __syncthreads();
    const int PC = s_total;

    // 5a. the compact row of each band's first row (the expert's run start, then the valid rows of
    // the expert's bands before it in hand-out order: full bands in layout order, then partial bands
    // by valid rows descending, ties to the lower owner); with the offsets, return offsets, chunk
    // bases and each expert's run this is all the permute needs, so it is published here and the
    // permute copies rows while the rest of the plan is built. (Step 5 computes the same rows again
    // for band_item rather than reading them back.)
    auto full_crow = [&](int e, int fpre, int i) { return s_cbase[e] + (fpre + i) * tbM; };
    auto partial_crow = [&](int e, int rows_before) { return s_cbase[e] + s_fb[e] * tbM + rows_before; };
    for (int g = tid; g < G; g += PLAN_THREADS) {
        const int e = g / R, r = g % R, n = s_n[g];
        const int m0 = s_off[g] / tbM, nfull = n / tbM;
        int fpre = 0;
        for (int q = 0; q < r; ++q) fpre += s_n[e * R + q] / tbM;
        for (int i = 0; i < nfull; ++i) p.tile_crow[m0 + i] = full_crow(e, fpre, i);
        if (n > nfull * tbM) {  // one partial band
            const int valid = n - nfull * tbM;
            int rows_before = 0;  // rows of the expert's partial bands before this one
            for (int rh = 0; rh < R; ++rh) {
                const int vh = s_n[e * R + rh] % tbM;
                if (vh == 0 || rh == r) continue;
                rows_before += ((vh > valid) || (vh == valid && rh < r)) ? vh : 0;
            }
            p.tile_crow[m0 + nfull] = partial_crow(e, rows_before);
        }
    }
    for (int e = tid; e < E; e += PLAN_THREADS) {
        p.experts[8 * e + 4] = (s_load[e] + BM - 1) / BM;
        p.experts[8 * e + 7] = s_cbase[e];
    }
    if (tid == 0) p.meta[META_PC] = PC;
    __threadfence();
    __syncthreads();
    // (MOE_TEST_STALL_LAYOUT: never published, so that the permute's bounded wait runs out)
    if (tid == 0 && !(s.flags & MOE_TEST_STALL_LAYOUT))
        red_release_gpu_add(reinterpret_cast<uint32_t*>(p.meta + META_LAYOUT), 1u);

    // 5b. remote-first schedule, the largest transfers first: bands by valid rows, descending, ties
    // in layout order. The full bands come first, in layout order (position = full bands of the
    // groups before + index); each group's partial band (valid = n mod tbM) follows, ranked by
    // (tbM - valid, group) among the partial bands: a counting sort over the buckets tbM - valid,
    // the groups of one bucket in group order (inside a warp of 32 consecutive groups by a match
    // mask, across warps by per-warp bucket counts). G <= PLAN_THREADS: thread g holds group g.
    __shared__ int s_bcnt[PLAN_THREADS / 32][128];  // partial bands per (warp of groups, bucket)
    __shared__ int s_bbase[128];                    // first rank of each bucket
    int n_full;
    {
        const int g = tid;
        const int fb = (g < G) ? s_n[g] / tbM : 0;
        const int o = block_exclusive_scan(fb, s_warp, &s_total);
        if (g < G) s_fbp[g] = o;
        n_full = s_total;
    }
    for (int i = tid; i < (PLAN_THREADS / 32) * 128; i += PLAN_THREADS) s_bcnt[i >> 7][i & 127] = 0;
    __syncthreads();
    {
        const int w = tid >> 5, lane = tid & 31;
        const int pv = (tid < G) ? s_n[tid] % tbM : 0;
        const int pb = pv ? tbM - pv : -1;  // bucket 1 .. tbM-1: the largest partial bands first
        const unsigned same = __match_any_sync(0xffffffffu, pb);
        const int in_warp = __popc(same & ((1u << lane) - 1u));
        if (pb >= 0 && in_warp == 0) s_bcnt[w][pb] = __popc(same);
        __syncthreads();
        int tot = 0;
        if (tid < tbM)
            for (int x = 0; x < PLAN_THREADS / 32; ++x) tot += s_bcnt[x][tid];
        const int o = block_exclusive_scan(tid < tbM ? tot : 0, s_warp, &s_total);
        if (tid < tbM) s_bbase[tid] = o;
        __syncthreads();
        if (pb >= 0) {
            int rk = s_bbase[pb] + in_warp;
            for (int x = 0; x < w; ++x) rk += s_bcnt[x][pb];
            s_prank[tid] = rk;
        }
    }
    __syncthreads();

    for (int e = tid; e < E; e += PLAN_THREADS) {
        int rk = 0;
        for (int f = 0; f < E; ++f)
            rk += (s_load[f] > s_load[e]) || (s_load[f] == s_load[e] && f < e);
        s_erank[e] = rk;
    }
    __syncthreads();
    // hand-out positions and down-projection items of the experts before each one in rank order
    __shared__ int s_ibase_down[MAX_E], s_nitems;
    for (int e = tid; e < E; e += PLAN_THREADS) {
        int base = 0, down = 0;
        for (int f = 0; f < E; ++f)
            if (s_erank[f] < s_erank[e]) {
                base += s_mt[f];
                down += (s_load[f] + BM - 1) / BM;
            }
        s_ebase[e] = base;
        s_ibase_down[e] = down;
        if (s_erank[e] == E - 1) s_nitems = down + (s_load[e] + BM - 1) / BM;  // the last expert's end the list
        p.experts[8 * e + 2] = base;        // first hand-out position of the expert's bands
        p.experts[8 * e + 3] = s_erank[e];  // the expert's rank in the hand-out order
    }
    __syncthreads();

    // 5. tiles, destination rows, schedule positions and hand-out positions.
    // Hand-out order (the schedule re-sorted stably by expert): experts one after another in rank
    // order (most loaded first); inside an expert its full bands in layout order, then its partial
    // bands by valid rows descending (ties to the lower owner), i.e. key (expert rank, -valid,
    // owner, row). A band's compact rows start after the valid rows of the expert's bands before it
    // in hand-out order: full bands fill whole tiles from the run's start, partial bands follow.
    // band_item: the down-projection item holding the band's last row, i.e. the item whose tiles
    // complete the band (its rows lie in this item and possibly the one before it of its expert),
    // read by the epilogue and the copy engines to tell the bands that the epilogue returns itself
    // (MOE_DIRECT_TAIL): a band is returned that way when this item is in the direct window, so no
    // band completed by the last wave is left to the copy engines.
    auto band_item_of = [&](int e, int crow, int valid) { return s_ibase_down[e] + (crow + valid - 1 - s_cbase[e]) / BM; };
    for (int g = tid; g < G; g += PLAN_THREADS) {
        const int e = g / R, r = g % R, n = s_n[g];
        const int m0 = s_off[g] / tbM;
        const int nt = (n + tbM - 1) / tbM, nfull = n / tbM;
        int fpre = 0;
        for (int q = 0; q < r; ++q) fpre += s_n[e * R + q] / tbM;
        int rbase = r * slice;  // owner r's rows of the experts before e (ret_off, from shared memory)
        for (int f = 0; f < e; ++f) rbase += s_n[f * R + r];
        for (int i = 0; i < nt; ++i) {
            const int m = m0 + i;
            const int valid = min(tbM, n - i * tbM);
            p.tiles[4 * m + 0] = e;
            p.tiles[4 * m + 1] = r;
            p.tiles[4 * m + 2] = s_off[g] + i * tbM;
            p.tiles[4 * m + 3] = valid;
            p.tile_ret[m] = rbase + i * tbM;
            if (mirror) s_tg[m] = g;
            if (i < nfull) {
                p.band_item[m] = band_item_of(e, full_crow(e, fpre, i), valid);
                p.sched[s_fbp[g] + i] = m;
                p.order[s_ebase[e] + fpre + i] = m;
                if (mirror) s_order[s_ebase[e] + fpre + i] = m;
            }
        }
        if (nt > nfull) {  // one partial band
            const int valid = n - nfull * tbM;
            int pos = 0, rows_before = 0;  // partial bands of the expert before this one, their rows
            for (int rh = 0; rh < R; ++rh) {
                const int vh = s_n[e * R + rh] % tbM;
                if (vh == 0 || rh == r) continue;
                const bool before = (vh > valid) || (vh == valid && rh < r);
                pos += before;
                rows_before += before ? vh : 0;
            }
            p.band_item[m0 + nfull] = band_item_of(e, partial_crow(e, rows_before), valid);
            p.order[s_ebase[e] + s_fb[e] + pos] = m0 + nfull;
            if (mirror) s_order[s_ebase[e] + s_fb[e] + pos] = m0 + nfull;
            p.sched[n_full + s_prank[g]] = m0 + nfull;
        }
    }
    __syncthreads();
    __threadfence_block();
    auto order_at = [&](int pos) { return mirror ? s_order[pos] : p.order[pos]; };
    auto group_of = [&](int m) { return mirror ? s_tg[m] : p.tiles[4 * m] * R + p.tiles[4 * m + 1]; };

    // 6. segments: runs of hand-out positions holding adjacent bands of one group, cut into pieces
    // of mgb bands
    for (int q = tid; q < MT; q += PLAN_THREADS) {
        auto adjacent = [&](int a, int b) {  // same group, consecutive bands (rows tbM apart)
            const int ma = order_at(a), mb = order_at(b);
            return mb == ma + 1 && group_of(ma) == group_of(mb);
        };
        int start = q;
        while (start > 0 && adjacent(start - 1, start)) --start;
        int end = q + 1;
        while (end < MT && adjacent(end - 1, end)) ++end;
        const int first = start + ((q - start) / s.mgb) * s.mgb;
        p.seg[2 * q + 0] = first;
        p.seg[2 * q + 1] = min(s.mgb, end - first);
    }

    // 7. GEMM work items: each expert's compact run cut into BM-row items (first compact row,
    // expert). The SwiGLU GEMM takes them with the experts in id order; the down-projection takes
    // the same items with the experts in hand-out order (rank order), so its item list is the SwiGLU
    // list re-ordered by expert. The down-projection's output rows go to the owner-aligned bands of
    // Yp, each band counted complete when all its rows of every N tile have been stored.
    for (int e = tid; e < E; e += PLAN_THREADS) {
        const int down = s_ibase_down[e], iu = (s_load[e] + BM - 1) / BM;
        p.experts[8 * e + 4] = iu;
        p.experts[8 * e + 5] = s_cbase[e] / BM;
        p.experts[8 * e + 6] = down;
        p.experts[8 * e + 7] = s_cbase[e];
        if (s_cbase[e] / BM + iu <= s.IU_max && down + iu <= s.MT_max)
            for (int i = 0; i < iu; ++i) {
                p.items_up[2 * (s_cbase[e] / BM + i)] = s_cbase[e] + i * BM;
                p.items_up[2 * (s_cbase[e] / BM + i) + 1] = e;
                p.items_down[2 * (down + i)] = s_cbase[e] + i * BM;
                p.items_down[2 * (down + i) + 1] = e;
            }
    }
    const int items = s_nitems;

    // 8. per-call meta, flags and trace reset
    if (tid == 0) {
        p.meta[META_P] = P;
        p.meta[META_MTILES] = MT;
        p.meta[META_UNITS] = copy_unit_count(s, MT);
        p.meta[META_ITEMS] = items;
        p.meta[META_ITEMS_UP] = PC / BM;
        p.meta[META_PC] = PC;
        p.meta[META_QUEUE] = 0;
        p.meta[META_QUEUE_SEQ] = 0;
        p.meta[META_TILES_UP] = 0;
        p.meta[META_TILES_DOWN] = 0;
        p.meta[META_DISPATCH] = 0;
        // MOE_TEST_PLAN_FAIL: report a failed check (detail -3) so that tests can see the status
        // reach the caller; the plan itself is still complete and valid
        const bool hook = (s.flags & MOE_TEST_PLAN_FAIL) != 0;
        const bool bad = P > s.P_max || PC > s.PC_max || hook;
        if (bad) set_status(p.meta, ST_BAD_PLAN, hook ? -3 : P > s.P_max ? P : PC);
    }
    if (tid < TR_STEP) p.trace[tid] = (tid == MOE_TRACE_GEMM2_START || tid == MOE_TRACE_COPY_START) ? ~0ull : 0ull;
    if (tid == 0 && p.host_rec) {  // moe_forward_dma: the band count for the host, then the call's tag
        p.host_rec[1] = (uint32_t)MT;
        p.host_rec[2] = (uint32_t)P;
        __threadfence_system();
        st_release_sys(p.host_rec, s.host_epoch);
    }
    const int nflags = min(MT, s.MT_max) * s.n_tiles_n2;
    for (int i = tid; i < nflags; i += PLAN_THREADS) p.flags[i] = 0u;
    for (int i = tid; i < min(MT, s.MT_max); i += PLAN_THREADS) p.bands[i] = 0u;
    for (int e = tid; e < E; e += PLAN_THREADS) {
        p.xrows[e] = 0u;
        p.xready[e] = 0u;
    }
}

cudaError_t launch_plan(const Shape& s, const PlanPtrs& p, cudaStream_t st) {
    const size_t smem = (s.MT_max <= PLAN_SMEM_TILES) ? (size_t)s.MT_max * 2 * sizeof(int) : 0;
    if (smem > 0) {
        const cudaError_t e =
            cudaFuncSetAttribute(reinterpret_cast<const void*>(&plan_kernel), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_k(plan_kernel, dim3(1), dim3(PLAN_THREADS), smem, st, true, s, p);
}

// ---------------------------------------------------------------------------------------------
// permute_kernel: one warp per work item. Items [0, T): token t computes its k slots (padded
// layout), compact slots (the compact row of its band's first row plus its row inside the band) and
// return slots, records t as the token and the padded row as the Yp row of its k compact rows, and
// copies x[t] into those rows of Xc: each lane first loads up to 16 vectors of 16 bytes (all loads
// in flight together), then stores them to the k rows. Items [T, T + E * BM/8): one group of 8 rows
// of an expert's last BM-row tile in the compact layout, marking those rows past the expert's rows
// as padding (token -1, no Yp row) and zeroing them. With x == nullptr only the slots, tokens and
// Yp rows are written. The kernel runs beside the second half of the plan kernel: each block waits
// for the row layout the plan publishes part-way through (see below), not for the plan's end.
// ---------------------------------------------------------------------------------------------
constexpr int PERM_VEC = 16;  // 16-byte vectors per lane per pass

__global__ void __launch_bounds__(256) permute_kernel(Shape s, const __nv_bfloat16* __restrict__ x, PlanPtrs p) {
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    // The first token's row does not depend on the plan: its loads are issued before the wait for
    // the plan kernel (while it runs), the rest of the work after.
    const int item0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    // nor do the first token's experts and ranks (the routing kernel completed before this grid
    // started): their loads overlap the wait too
    int e0 = 0, rk0 = 0;
    if (item0 < s.T && lane < s.k) {
        e0 = p.idx[(size_t)item0 * s.k + lane];
        rk0 = p.rank[(size_t)item0 * s.k + lane];
    }
    const int vec0 = s.d / 8;
    uint4 v[PERM_VEC];  // one pass of a row: the first token's first pass is loaded here
    const bool prefetched = x != nullptr && item0 < s.T;
    if (prefetched) {
        const uint4* xs0 = reinterpret_cast<const uint4*>(x) + (size_t)item0 * vec0;
#pragma unroll
        for (int i = 0; i < PERM_VEC; ++i) {
            const int vi = i * 32 + lane;
            if (vi < vec0) v[i] = __ldg(xs0 + vi);
        }
    }
    // This grid starts once the plan kernel has passed its own wait for the routing kernel,
    // so the routing outputs are complete. The plan's layout (offsets, return offsets, chunk bases,
    // the bands' compact rows, each expert's run) is published part-way through the plan with a
    // release; thread 0's acquire and the barrier order every thread's later loads after it, and no
    // thread of this grid reads those tables before. The next launch reads the rest of the plan from
    // its prologue on, so it may start only after the plan kernel has completed: every block but the
    // last lets it start at once, the last block only after waiting for the plan kernel; it can start
    // only once every block has done so, and this grid completes after the plan. (The last block is
    // normally the last to start, so it rarely waits; the start order matters for speed only.)
    __shared__ int s_layout;
    const bool last = blockIdx.x == gridDim.x - 1;
    if (threadIdx.x == 0) {
        const bool ok = wait_word(reinterpret_cast<const uint32_t*>(p.meta + META_LAYOUT), s.timeout_ns);
        if (!ok) set_status(p.meta, ST_LAYOUT_TIMEOUT, 0);
        if (last) griddep_wait();
        s_layout = ok;
    }
    __syncthreads();
    if (!last || threadIdx.x == 0) griddep_launch();
    if (!s_layout) return;
    const int PC = p.meta[META_PC];
    const int per = s.T / s.R, slice = per * s.k, E = s.E, R = s.R, k = s.k;
    const int vec = s.d / 8;  // 16-byte vectors per row
    const uint4* xs = reinterpret_cast<const uint4*>(x);
    uint4* xc = reinterpret_cast<uint4*>(p.Xc);
    const bool ok_pc = PC >= 0 && PC <= s.PC_max;
    const int groups = BM / 8;
    const int pad_items = ok_pc ? E * groups : 0;

    for (int item = item0; item < s.T + pad_items; item += nwarps) {
        if (item < s.T) {
            const int t = item, r = t / per, c = t / s.chunk_tokens;
            int my_cs = 0, my_y = 0;
            if (lane < k) {
                const bool first = item == item0;
                const int e = first ? e0 : p.idx[(size_t)t * k + lane];
                const int rk = p.chunk_base[(size_t)c * E + e] + (first ? rk0 : p.rank[(size_t)t * k + lane]);
                my_y = p.offsets[e * R + r] + rk;
                const int m = my_y / s.tbM;  // bands start at multiples of the tile height
                my_cs = (m >= 0 && m < s.MT_max) ? p.tile_crow[m] + (my_y - m * s.tbM) : -1;
                p.slot[(size_t)t * k + lane] = my_y;
                p.cslot[(size_t)t * k + lane] = my_cs;
                p.ret_slot[(size_t)t * k + lane] = r * slice + p.ret_off[r * (E + 1) + e] + rk;
            }
            int cs[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) cs[j] = __shfl_sync(0xffffffffu, my_cs, j);
            bool good = ok_pc;
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < k) good &= (cs[j] >= 0 && cs[j] < PC);
            if (!good) {
                if (lane == 0) set_status(p.meta, ST_BAD_PLAN, t);
                continue;
            }
            if (lane < k) {
                p.tok_of[my_cs] = t;    // the compact row's token (read by a fused dispatch)
                p.yrow[my_cs] = my_y;   // and its output row (read by the down-projection's epilogue)
            }
            if (xs == nullptr) continue;  // plan only: slots without the row copy
            for (int base = 0; base < vec; base += 32 * PERM_VEC) {
                if (!(prefetched && item == item0 && base == 0)) {
#pragma unroll
                    for (int i = 0; i < PERM_VEC; ++i) {
                        const int vi = base + i * 32 + lane;
                        if (vi < vec) v[i] = __ldg(xs + (size_t)t * vec + vi);
                    }
                }
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j >= k) break;
#pragma unroll
                    for (int i = 0; i < PERM_VEC; ++i) {
                        const int vi = base + i * 32 + lane;
                        if (vi < vec) xc[(size_t)cs[j] * vec + vi] = v[i];
                    }
                }
            }
        } else {
            // the expert's run is [cb, cb + iu * BM) and holds `rows` real rows
            const int q = item - s.T, e = q / groups, g = q % groups;
            const int iu = p.experts[8 * e + 4], cb = p.experts[8 * e + 7];
            int rows = 0;
            for (int r = 0; r < R; ++r) rows += p.counts[e * R + r];
            if (iu <= 0) continue;
            const uint4 z = make_uint4(0, 0, 0, 0);
            for (int rr = max(rows, (iu - 1) * BM + g * 8); rr < (iu - 1) * BM + (g + 1) * 8; ++rr) {
                const size_t row = (size_t)cb + rr;
                if (row >= (size_t)PC) break;
                if (lane == 0) {  // a padding row: zeros
                    p.tok_of[row] = -1;
                    p.yrow[row] = -1;
                }
                if (xs == nullptr) continue;
                for (int v = lane; v < vec; v += 32) xc[row * vec + v] = z;
            }
        }
    }
}

cudaError_t launch_permute(const Shape& s, const __nv_bfloat16* x, const PlanPtrs& p, int sms, cudaStream_t st) {
    const int items = s.T + s.E * (BM / 8);
    const int blocks = min((items + 7) / 8, sms * 16);
    return launch_k(permute_kernel, dim3(blocks), dim3(256), 0, st, true, s, x, p);
}

}  // namespace moe
