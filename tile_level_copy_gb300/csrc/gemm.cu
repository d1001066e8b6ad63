// Persistent grouped expert GEMMs on tcgen05 (UMMA 128 x N x 16, fp32 accumulators in TMEM),
// fed by TMA through a 4-stage shared-memory ring, with warp-specialised roles:
//   warp 0      one thread issues the TMA loads of A (token rows) and B (expert weights)
//   warp 1      allocates 512 TMEM columns; one thread issues the UMMAs (two accumulators, so the
//               epilogue of tile i overlaps the main loop of tile i+1)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, conversion, staging in shared memory and
//               TMA tensor stores of 32 x 32 chunks to global memory
//
// Method: "Fine-grained Computation-Communication Overlap via Tile-level Signaling and Scheduling
// for Mixture-of-Experts" (pith.science/paper/W2ZARMHG):
//   "Core claim" - one rank-wide persistent GEMM covers all experts in one launch and publishes a
//       readiness flag after each tile's epilogue store;
//   "Load-bearing premise" and "Referee Report" major comment 2 (§3.3.1) - the tile must be
//       visible before the flag: each of the four epilogue warps waits until its TMA stores of the
//       tile have completed, fences the async proxy, then adds 1 to the tile flag with
//       red.release.gpu; the consumer reads the flag with ld.acquire.gpu (ready at 4) and fences
//       the async proxy before its bulk copy.
//   "What carries the argument" - the consumer runs on a small dedicated SM partition; here the
//       partition is the last consumer_ctas CTAs of the same cooperative launch, so producers and
//       consumers are guaranteed to be co-resident.
#include "copy_ring.cuh"

namespace moe {

struct Smem {
    uint8_t* stages;
    uint8_t* epi;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    uint64_t* cbar;
    uint32_t* tmem_base;
    volatile int* abort;
    volatile int* unit;
    int* tab;  // [cum (E+1) | first (E) | count (E)]
};

__device__ __forceinline__ Smem carve_smem(uint8_t* raw) {
    Smem sm;
    const uint32_t a = smem_u32(raw);
    uint8_t* base = raw + (((a + 1023u) & ~1023u) - a);
    sm.stages = base;
    sm.epi = base + STAGES * STAGE_BYTES;
    uint8_t* misc = sm.epi + EPI_BYTES;
    sm.full = reinterpret_cast<uint64_t*>(misc);
    sm.empty = sm.full + STAGES;
    sm.acc_full = sm.empty + STAGES;
    sm.acc_empty = sm.acc_full + 2;
    sm.drain = sm.acc_empty + 2;
    sm.cbar = sm.drain + 1;
    sm.tmem_base = reinterpret_cast<uint32_t*>(sm.cbar + COPY_NBUF);
    sm.abort = reinterpret_cast<volatile int*>(sm.tmem_base + 1);
    sm.unit = sm.abort + 1;
    sm.tab = const_cast<int*>(sm.unit + 2);
    return sm;
}

// One GEMM tile: work item (mA, mB) x N tile n of expert e. Rows 0-63 of the UMMA tile come from
// row rowA on, rows 64-127 from row rowB on (rowB = rowA + 64 when the item is a single band).
// mB == mA: one band of 128 rows; mB == -1: one band of 64 rows alone; otherwise two half bands.
struct TileRef {
    int mA, mB, n, e, rowA, rowB;
};

__device__ __forceinline__ TileRef make_ref(int mA, int mB, int n, const int32_t* tiles) {
    TileRef r;
    r.mA = mA;
    r.mB = mB;
    r.n = n;
    r.e = tiles[4 * mA + 0];
    r.rowA = tiles[4 * mA + 2];
    r.rowB = (mB >= 0 && mB != mA) ? tiles[4 * mB + 2] : r.rowA + 64;
    return r;
}

// SwiGLU GEMM order: expert-major; inside an expert, N tiles outer and work items inner, so the
// CTAs working at the same time share each weight tile through L2.
// tab = [cum (E+1) | first item (E) | items (E)]
__device__ __forceinline__ TileRef decode_up(int t, const int* tab, int E, const int32_t* items,
                                             const int32_t* tiles) {
    const int* cum = tab;
    const int* first = tab + (E + 1);
    const int* count = first + E;
    int lo = 0, hi = E - 1;  // largest e with cum[e] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int e = lo, local = t - cum[e], cnt = count[e];
    const int n = local / cnt, it = first[e] + local % cnt;
    return make_ref(items[2 * it], items[2 * it + 1], n, tiles);
}

// Down-projection order: work items in schedule (remote-first) order, all N tiles of an item together.
__device__ __forceinline__ TileRef decode_down(int t, int nN, const int32_t* items, const int32_t* tiles) {
    const int it = t / nN;
    return make_ref(items[2 * it], items[2 * it + 1], t - it * nN, tiles);
}

template <int MODE>  // 1: SwiGLU up-projection -> Hp; 2: down-projection -> Yp (+ flags / consumer)
__global__ void __launch_bounds__(GEMM_THREADS_MAX, 1)
    gemm_kernel(Shape s, PlanPtrs p, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAh,
                const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                const __grid_constant__ CUtensorMap tmOut, int num_producers, int overlapped) {
    extern __shared__ uint8_t smem_raw[];
    Smem sm = carve_smem(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const bool producer = (int)blockIdx.x < num_producers;

    int MT = p.meta[META_MTILES], NI = p.meta[META_ITEMS];
    if (MT < 0 || MT > s.MT_max || NI < 0 || NI > MT) MT = NI = 0;
    const int nN = (MODE == 1) ? s.ffn / BN1 : s.n_tiles_n2;
    const int BN = (MODE == 1) ? 2 * BN1 : s.bn2;  // UMMA N
    const int KB = ((MODE == 1) ? s.d : s.ffn) / BK;
    const int total = NI * nN;
    const uint32_t tx_bytes = A_STAGE_BYTES + BN * BK * 2;
    const unsigned long long tmo = s.timeout_ns;

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.acc_full[i], 1);
            mbar_init(&sm.acc_empty[i], 128);
        }
        mbar_init(sm.drain, 1);
        for (int i = 0; i < COPY_NBUF; ++i) mbar_init(&sm.cbar[i], 1);
        *sm.abort = 0;
        mbar_fence_init();
    }
    if (MODE == 1) {
        for (int e = tid; e < s.E; e += blockDim.x) {
            sm.tab[(s.E + 1) + e] = p.experts[8 * e + 5];         // first work item
            sm.tab[(s.E + 1) + s.E + e] = p.experts[8 * e + 4];   // work items
        }
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int e = 0; e < s.E; ++e) {
                sm.tab[e] = acc;
                acc += sm.tab[(s.E + 1) + s.E + e] * nN;
            }
            sm.tab[s.E] = acc;
        }
    }
    if (producer && warp == 1) {
        tmem_alloc(sm.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (producer && tid == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmAh);
        tma_prefetch_desc(&tmB0);
        tma_prefetch_desc(&tmOut);
        if (MODE == 1) tma_prefetch_desc(&tmB1);
        if (MODE == 2) atomicMin(&p.trace[MOE_TRACE_GEMM2_START], globaltimer());
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = producer ? *sm.tmem_base : 0u;
    unsigned long long last_end = 0;
    const uint32_t want = FLAG_READY * s.n_tiles_n2 + ((s.flags & MOE_TEST_STALL_CONSUMER) ? 1u : 0u);

    // Extra warps (launched with MOE_COPY_WARPS): SIMT copy engines beside the GEMM warps.
    if (warp >= GEMM_WARPS) {
        if (MODE == 2 && overlapped) copy_units_simt(s, p, sm.abort, META_QUEUE, want);
        return;
    }

    if (producer) {
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer ----------------
            int st = 0;
            uint32_t ph = 0, issued = 0, last_ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += num_producers) {
                const TileRef tr = (MODE == 1) ? decode_up(t, sm.tab, s.E, p.items_up, p.tiles)
                                               : decode_down(t, nN, p.items_down, p.tiles);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&sm.empty[st], ph ^ 1u, tmo, sm.abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.full[st], tx_bytes);
                    uint8_t* a = sm.stages + st * STAGE_BYTES;
                    uint8_t* b = a + A_STAGE_BYTES;
                    if (tr.mB >= 0 && tr.mB != tr.mA) {  // two half bands: two 64-row boxes
                        tma_load_2d(a, &tmAh, &sm.full[st], kb * BK, tr.rowA);
                        tma_load_2d(a + A_STAGE_BYTES / 2, &tmAh, &sm.full[st], kb * BK, tr.rowB);
                    } else {
                        tma_load_2d(a, &tmA, &sm.full[st], kb * BK, tr.rowA);
                    }
                    if (MODE == 1) {
                        tma_load_3d(b, &tmB0, &sm.full[st], kb * BK, tr.n * BN1, tr.e);
                        tma_load_3d(b + BN1 * BK * 2, &tmB1, &sm.full[st], kb * BK, tr.n * BN1, tr.e);
                    } else {
                        tma_load_3d(b, &tmB0, &sm.full[st], kb * BK, tr.n * BN, tr.e);
                    }
                    issued |= 1u << st;
                    last_ph = (last_ph & ~(1u << st)) | (ph << st);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 0);
                *sm.abort = 1;
                int never = 0;
                for (int i = 0; i < STAGES; ++i)  // let loads in flight land before the CTA leaves
                    if (issued & (1u << i)) mbar_wait(&sm.full[i], (last_ph >> i) & 1u, tmo, &never);
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------- UMMA issuer ----------------
            const uint32_t idesc = umma_idesc_bf16(BM, BN);
            int st = 0, b = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true, any = false;
            for (int t = blockIdx.x; t < total && ok; t += num_producers) {
                if (!mbar_wait(&sm.acc_empty[b], aph ^ 1u, tmo, sm.abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(b * 256);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&sm.full[st], ph, tmo, sm.abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sm.stages + st * STAGE_BYTES);
                    const uint64_t ad = sdesc_sw128(a_addr);
                    const uint64_t bd = sdesc_sw128(a_addr + A_STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes along K per UMMA_K = 16
                        umma_bf16(dt, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    umma_commit(&sm.empty[st]);
                    any = true;
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&sm.acc_full[b]);
                b ^= 1;
                if (b == 0) aph ^= 1u;
            }
            if (!ok) {
                if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 1);
                *sm.abort = 1;
                if (any) {  // wait for the UMMAs in flight before TMEM is released
                    int never = 0;
                    umma_commit(sm.drain);
                    mbar_wait(sm.drain, 0, tmo, &never);
                }
            }
        } else if (warp >= 2) {
            // ---------------- epilogue ----------------
            // Each warp owns TMEM lanes 32q..32q+31 (tile rows). Per 32-column chunk: tcgen05.ld,
            // convert, write the 32 x 32 bf16 chunk to a shared staging buffer (each lane its row,
            // 16-byte pieces in a lane-rotated order, free of bank conflicts), then lane 0 issues one
            // TMA tensor store of the chunk. Two staging buffers per warp alternate.
            const int q = warp & 3;  // TMEM lane quarter this warp may access
            const bool flags = (MODE == 2) && overlapped;
            uint8_t* ebuf = sm.epi + (warp - 2) * 2 * EPI_CHUNK_BYTES;
            int eb = 0;
            int b = 0;
            uint32_t aph = 0;
            auto stage_chunk = [&](const uint32_t (&pk)[16], int x, int y) {
                if (lane == 0) bulk_wait_read_1();  // the store that last used this buffer has read it
                __syncwarp();
                uint4* dst = reinterpret_cast<uint4*>(ebuf + eb * EPI_CHUNK_BYTES + lane * (EPI_CHUNK * 2));
                const uint4 u0 = make_uint4(pk[0], pk[1], pk[2], pk[3]), u1 = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                const uint4 u2 = make_uint4(pk[8], pk[9], pk[10], pk[11]);
                const uint4 u3 = make_uint4(pk[12], pk[13], pk[14], pk[15]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int pi = (i + lane) & 3;
                    dst[pi] = pi == 0 ? u0 : pi == 1 ? u1 : pi == 2 ? u2 : u3;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmOut, ebuf + eb * EPI_CHUNK_BYTES, x, y);
                    bulk_commit();
                }
                eb ^= 1;
            };
            for (int t = blockIdx.x; t < total; t += num_producers) {
                const TileRef tr = (MODE == 1) ? decode_up(t, sm.tab, s.E, p.items_up, p.tiles)
                                               : decode_down(t, nN, p.items_down, p.tiles);
                if (!mbar_wait(&sm.acc_full[b], aph, tmo, sm.abort)) {
                    if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 2);
                    *sm.abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * 256);
                // rows 0-63 belong to band mA, rows 64-127 to band mB (or to mA for a 128-row band)
                const int mq = (q < 2) ? tr.mA : tr.mB;
                const bool active = mq >= 0;
                const int y = (q < 2 ? tr.rowA : tr.rowB) + (q & 1) * 32;
                const uint32_t inc = (tr.mB == tr.mA) ? 1u : 2u;  // quarters per band: 4 in all
                if (MODE == 1) {
#pragma unroll 1
                    for (int c = 0; c < BN1 / 32; ++c) {
                        uint32_t g[32], u[32];
                        tmem_ld32(tb + c * 32, g);
                        tmem_ld32(tb + BN1 + c * 32, u);
                        if (active) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                                const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * __uint_as_float(u[2 * i]);
                                const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * __uint_as_float(u[2 * i + 1]);
                                pk[i] = pack_bf16x2(h0, h1);
                            }
                            stage_chunk(pk, tr.n * BN1 + c * 32, y);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tb + c * 32, v);
                        if (active) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                            stage_chunk(pk, tr.n * BN + c * 32, y);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&sm.acc_empty[b]);
                if (MODE == 2 && active) {
                    if (flags) {
                        // Publish this warp's rows of the tile: its TMA stores must be complete (not
                        // only read out of shared memory), the async proxy fenced against the generic
                        // one, then lane 0 adds its share (1 for a quarter of a 128-row band, 2 for
                        // half of a 64-row one) to the tile's flag with release semantics (the tile
                        // is ready at 4) and to its band's counter (the band is ready at 4 x tiles
                        // per band), which is what consumers poll.
                        if (lane == 0) {
                            bulk_wait_all();
                            fence_proxy_async_global();
                            __threadfence();
                            red_release_gpu_add(p.flags + (size_t)mq * s.n_tiles_n2 + tr.n, inc);
                            const uint32_t before = atom_release_gpu_add(p.bands + mq, inc);
                            if (before + inc == FLAG_READY * (uint32_t)s.n_tiles_n2)
                                atomicMax(&p.trace[MOE_TRACE_BAND_DONE], globaltimer());
                        }
                        __syncwarp();
                    }
                    if (lane == 0) last_end = globaltimer();
                }
                b ^= 1;
                if (b == 0) aph ^= 1u;
            }
            if (lane == 0) bulk_wait_all();  // staging buffers stay valid until every store is done
            __syncwarp();
        }
    }
    tc_fence_before();
    named_bar_sync(1, GEMM_THREADS);  // the GEMM warps only: extra copy warps run on independently
    if (producer && warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    if (MODE == 2 && producer && warp >= 2 && lane == 0 && last_end)
        atomicMax(&p.trace[MOE_TRACE_GEMM2_END], last_end);

    if (MODE == 2 && overlapped && (!producer || (s.flags & MOE_TAIL_ASSIST)))
        copy_units(s, p, sm.stages, sm.cbar, sm.abort, META_QUEUE, true, want);
}

static cudaError_t set_smem_attr(const void* fn) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
}

cudaError_t launch_gemm_swiglu(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA, const CUtensorMap& tmAh,
                               const CUtensorMap& tmW1, const CUtensorMap& tmW3, const CUtensorMap& tmOut, int sms,
                               cudaStream_t st) {
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(&gemm_kernel<1>));
    if (e != cudaSuccess) return e;
    gemm_kernel<1><<<sms, GEMM_THREADS, GEMM_SMEM, st>>>(s, p, tmA, tmAh, tmW1, tmW3, tmOut, sms, 0);
    return cudaGetLastError();
}

cudaError_t launch_gemm_down(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA, const CUtensorMap& tmAh,
                             const CUtensorMap& tmW2, const CUtensorMap& tmOut, int sms, int consumers, bool overlapped,
                             cudaStream_t st) {
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(&gemm_kernel<2>));
    if (e != cudaSuccess) return e;
    const int producers = overlapped ? sms - consumers : sms;
    int ov = overlapped ? 1 : 0;
    const int threads = (overlapped && (s.flags & MOE_COPY_WARPS)) ? GEMM_THREADS_MAX : GEMM_THREADS;
    Shape sa = s;
    PlanPtrs pa = p;
    CUtensorMap a = tmA, ah = tmAh, b0 = tmW2, b1 = tmW2, o = tmOut;
    if (!overlapped) {
        gemm_kernel<2><<<sms, GEMM_THREADS, GEMM_SMEM, st>>>(sa, pa, a, ah, b0, b1, o, producers, ov);
        return cudaGetLastError();
    }
    // Cooperative launch: every CTA (producers and consumers) is resident at once, or the launch
    // fails; the consumers' waits on producer flags can therefore always be satisfied.
    void* args[] = {&sa, &pa, &a, &ah, &b0, &b1, &o, (void*)&producers, &ov};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&gemm_kernel<2>), dim3(sms), dim3(threads),
                                       args, GEMM_SMEM, st);
}

// Sequential return copy: every SM takes copy units, no flags ([TLS Figure 9 caption] baseline).
__global__ void __launch_bounds__(GEMM_THREADS, 1) copy_seq_kernel(Shape s, PlanPtrs p) {
    extern __shared__ uint8_t smem_raw[];
    Smem sm = carve_smem(smem_raw);
    if (threadIdx.x == 0) {
        for (int i = 0; i < COPY_NBUF; ++i) mbar_init(&sm.cbar[i], 1);
        *sm.abort = 0;
        mbar_fence_init();
    }
    __syncthreads();
    copy_units(s, p, sm.stages, sm.cbar, sm.abort, META_QUEUE_SEQ, false, 0u);
}

cudaError_t launch_copy_seq(const Shape& s, const PlanPtrs& p, int sms, cudaStream_t st) {
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(&copy_seq_kernel));
    if (e != cudaSuccess) return e;
    copy_seq_kernel<<<sms, GEMM_THREADS, GEMM_SMEM, st>>>(s, p);
    return cudaGetLastError();
}

}  // namespace moe
