// The small-problem kernel: one output tile per cluster, no persistent loop.
//
// A problem with fewer 256×256 tiles than the GPU has CTA pairs is latency
// bound: its time is the launch, the set-up, the first operand loads from
// DRAM, a short main loop, the epilogue and the teardown, not tensor-core
// work.  The persistent kernel's path through those steps is long (six warps
// in three roles, a 512-column double-buffered accumulator, a 230 KB ring and
// staging buffer, a shared-memory staged TMA store, a work schedule).  This
// kernel has the shortest path the same hardware steps allow, and narrow tiles
// so that such a problem covers many SMs:
//   - one 128·CG × BN tile of C per cluster (CG = 1: one CTA, cta_group::1
//     MMAs of 128×BN; CG = 2: a CTA pair, cta_group::2 MMAs of 256×BN with
//     each CTA loading its 128 rows of A and BN/2 rows of B);
//   - four warps: lane 0 of warp 0 issues the TMA loads of every k-block
//     through an S-stage ring, warp 1 (of the pair's first CTA) runs the MMA
//     loop with one elected lane issuing, then all four warps drain the accumulator — warp w
//     reads tensor-memory lanes 32w..32w+31, which are rows of the tile — and
//     store their rows of C straight from registers, 16 bytes at a time;
//   - tensor memory: BN columns, one accumulator; shared memory: the ring;
//   - with few tiles and deep k, each tile's k range is cut into `pieces`
//     equal pieces on consecutive clusters (split-K): the first piece owns
//     the tile; the others write their fp32 partial tiles to the workspace
//     and publish per-warp flags tagged with the launch's id, and the owner
//     adds them to its own accumulator in piece order (k order) before the
//     rounding, so results do not depend on timing.
// A and B are K-major ([M, K] and [N, K] rows); the accumulator is fp32 and the
// result fp16 or bf16, rounded to nearest even, as in the persistent kernel.
// The operation and the tile loop are those of the Tilus tutorial's kernels
// ("3. Warp Specialization", §The Full Kernel: a producer filling a stage ring
// and a consumer issuing the MMAs, one tile per thread block), on tcgen05.
//
// Every wait is bounded as in the persistent kernel (the same watchdog word,
// sites and limits); on expiry the CTA stops, lets its copies and MMAs in
// flight finish (bounded), frees its tensor memory and exits.

#pragma once

#include "persistent.cuh"   // tile constants, the watchdog and its waits, descriptors

namespace g16 {

constexpr int kSmallThreads = 128;   // 4 warps: producer lane, MMA lane, then all four drain

template <int CG, int BN, int STAGES, bool BF = false, bool SPLIT = false>
struct SCfg {
    static constexpr int kCG = CG;
    static constexpr bool kSplit = SPLIT;            // split-K: the launch's tiles are cut into pieces
    static constexpr int kBN = BN;
    static constexpr int kStages = STAGES;
    static constexpr bool kBF = BF;
    static constexpr int kTileM = kBlockM * CG;       // rows of C per tile
    static constexpr int kBRows = BN / CG;            // B rows this CTA loads per stage
    static constexpr int kABytes = kBlockM * kBlockK * 2;
    static constexpr int kBBytes = kBRows * kBlockK * 2;
    static constexpr int kTxBytes = (kABytes + kBBytes) * CG;   // per stage, on the first CTA's barrier
    static constexpr int kTmemCols = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
    static constexpr int kRingBytes = STAGES * (kABytes + kBBytes);
    static constexpr int kCtlBytes = 256;
    // split-K: each warp's scratch in the (idle by then) ring, and the most
    // pieces a tile whose partials fit in it at once (a power of two, <= 8)
    static constexpr int kScratchBytes = kRingBytes / 4;
    static constexpr int kPartialBytes = BN * 32 * 4;             // one warp's 32 rows x BN fp32
    static constexpr int kMaxPieces = (kScratchBytes / kPartialBytes + 1) >= 8 ? 8
                                    : (kScratchBytes / kPartialBytes + 1) >= 4 ? 4 : 2;
    static constexpr int kSmemBytes = 1024 + kRingBytes + kCtlBytes;
    // kind::f16 instruction descriptor: D fp32, A/B fp16 or bf16, both K-major,
    // N>>3 at bit 17, M>>4 at bit 24 (as in KCfg).
    static constexpr uint32_t kIdesc = (1u << 4) | (uint32_t(BF) << 7) | (uint32_t(BF) << 10) |
                                       (uint32_t(BN >> 3) << 17) | (uint32_t(kTileM >> 4) << 24);

    static_assert(CG == 1 || CG == 2, "one CTA or a CTA pair");
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 128, "the epilogue drains 32-column groups, at most 4");
    static_assert(kBRows % 8 == 0, "B rows per CTA must fill whole 8-row swizzle atoms");
    static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "stages stay 1 KB aligned");
    static_assert(kSmemBytes <= 232448, "dynamic shared memory limit per CTA");
    static_assert(kPartialBytes <= kScratchBytes, "a partial tile fits in a warp's scratch");
};

template <int STAGES>
struct SmallCtl {
    uint64_t full[STAGES];    // stage loaded (the first CTA's copy counts both CTAs' bytes)
    uint64_t empty[STAGES];   // stage consumed (each CTA's own copy)
    uint64_t acc_full;        // accumulator complete
    uint64_t mma_done;        // every MMA retired (teardown)
    uint64_t xfer[4];         // split-K: the other pieces' partials landed in a warp's scratch
    uint32_t tmem_base;
    uint32_t abort_flag;
};

struct SmallParams {
    CUtensorMap tmA;    // A: dims {K, M}, box {64, 128}
    CUtensorMap tmB;    // B: dims {K, N}, box {64, BN/CG}
    uint16_t* C;
    int64_t ldc;
    int32_t M;
    int32_t N;
    uint32_t m_tiles;   // tile t covers rows (t % m_tiles)·128·CG and columns (t / m_tiles)·BN
    uint32_t num_kb;
    uint64_t timeout_ns;
    uint64_t item_timeout_ns;
    uint32_t* watchdog;
    int32_t inject_stall;
    // split-K (pieces > 1): cluster c runs piece c % pieces of tile c / pieces
    uint32_t pieces;
    float* partials;       // [cluster][cta rank][warp][BN/4][32 rows] float4: a piece's partial tile
    uint64_t* flags;       // [cluster][cta rank][warp]: launch_id once that warp's partial is written
    uint64_t launch_id;    // unique per launch, so stale flags never match
};

template <class Cfg>
__global__ void __launch_bounds__(kSmallThreads, 1) gemm_f16_nt_small_kernel(const __grid_constant__ SmallParams p) {
    constexpr int CG = Cfg::kCG;
    constexpr int BN = Cfg::kBN;
    constexpr int S = Cfg::kStages;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // 128-byte swizzle atoms need 1 KB alignment
    const uint32_t sA = base;
    const uint32_t sB = sA + S * Cfg::kABytes;
    SmallCtl<S>* ctl = reinterpret_cast<SmallCtl<S>*>(smem_raw + (base - raw) + Cfg::kRingBytes);

    const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t prank = CG == 2 ? ptx::cluster_ctarank() : 0u;   // rank in the pair
    const uint32_t cluster = CG == 2 ? ptx::cluster_id_x() : blockIdx.x;

    const uint32_t full0 = ptx::smem_u32(&ctl->full[0]);
    const uint32_t empty0 = ptx::smem_u32(&ctl->empty[0]);
    const uint32_t acc_full = ptx::smem_u32(&ctl->acc_full);
    const uint32_t mma_done = ptx::smem_u32(&ctl->mma_done);

    // this cluster's tile and k-block range [kb0, kb1) (all of k without split-K)
    const uint32_t tile = Cfg::kSplit ? cluster / p.pieces : cluster;
    const uint32_t piece = Cfg::kSplit ? cluster - tile * p.pieces : 0u;
    const uint32_t kb0 = Cfg::kSplit ? p.num_kb * piece / p.pieces : 0u;
    const uint32_t kb1 = Cfg::kSplit ? p.num_kb * (piece + 1) / p.pieces : p.num_kb;
    const uint32_t nkb = kb1 - kb0;
    const uint32_t mt = tile % p.m_tiles, nt = tile / p.m_tiles;
    const int32_t m0 = int32_t(mt * Cfg::kTileM + prank * kBlockM);   // this CTA's first row
    const int32_t n0 = int32_t(nt * BN);                               // the tile's first column
    const int32_t b0 = n0 + int32_t(prank) * Cfg::kBRows;              // this CTA's first B row

    // The producer's k-block loads: stage s of the ring, k-block kb0 + i.
    auto load_stage = [&](uint32_t s, uint32_t i) {
        const uint32_t full_tgt = CG == 2 ? ptx::mapa(full0, 0) : full0;
        if (prank == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * s, uint32_t(Cfg::kTxBytes));
        const int32_t k0 = int32_t((kb0 + i) * kBlockK);
        const uint32_t bar = full_tgt + 8 * s;
        if constexpr (CG == 2) {
            ptx::tma_load_2d_pair(sA + s * Cfg::kABytes, &p.tmA, k0, m0, bar);
            ptx::tma_load_2d_pair(sB + s * Cfg::kBBytes, &p.tmB, k0, b0, bar);
        } else {
            ptx::tma_load_2d(sA + s * Cfg::kABytes, &p.tmA, k0, m0, bar);
            ptx::tma_load_2d(sB + s * Cfg::kBBytes, &p.tmB, k0, b0, bar);
        }
    };

    uint32_t pre = 0;   // k-blocks the producer issued before the CTA-wide sync
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);    // the first CTA's expect-tx arrive
            ptx::mbar_init(empty0 + 8 * s, 1);   // one tcgen05.commit
        }
        ptx::mbar_init(acc_full, 1);
        ptx::mbar_init(mma_done, 1);
        for (int q = 0; q < 4; ++q) ptx::mbar_init(ptx::smem_u32(&ctl->xfer[q]), 1);
        ctl->abort_flag = 0u;
        ptx::fence_mbarrier_init();
        // One CTA: the barriers are this thread's own, so it fills the empty
        // ring at once (after the previous kernel on the stream has completed),
        // while the others allocate tensor memory and meet at the sync.  A pair's
        // loads complete on the first CTA's barriers, which the cluster sync
        // must show to the other CTA first.
        if constexpr (CG == 1) {
            if (!p.inject_stall) {
                ptx::griddep_wait();
                pre = nkb < uint32_t(S) ? nkb : uint32_t(S);
                for (uint32_t i = 0; i < pre; ++i) load_stage(i, i);
            }
        }
    }
    if (warp == 0 && lane == 0 && pre == 0) {
        ptx::prefetch_tensormap(&p.tmA);
        ptx::prefetch_tensormap(&p.tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_u32(&ctl->tmem_base), Cfg::kTmemCols);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(&ctl->tmem_base);

    // Programmatic dependent launch, as in the persistent kernel: global
    // memory only after the previous kernel on the stream has completed.
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();

    Watch w;
    w.limit_ns = p.timeout_ns;
    w.abort_flag = &ctl->abort_flag;
    w.abort_addr = ptx::smem_u32(&ctl->abort_flag);
    w.ctas = CG;
    w.rank = prank;
    w.word = p.watchdog;
    Watch wi = w;   // waits that can span the whole main loop
    wi.limit_ns = p.item_timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && !p.inject_stall) {
            uint32_t issued = pre;
            bool ok = true;
            for (uint32_t i = pre; i < nkb; ++i) {
                const uint32_t s = i % uint32_t(S), ph = (i / uint32_t(S)) & 1u;
                // (a fresh barrier's phase of parity 1 counts as complete: no wait on the first pass)
                if (!wait(empty0 + 8 * s, ph ^ 1u, wi, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                load_stage(s, i);
                ++issued;
            }
            if (!ok && issued) {
                // Let the copies already issued land before the CTA can exit.
                if (prank == 0) {
                    const uint32_t n = issued < uint32_t(S) ? issued : uint32_t(S);
                    for (uint32_t i = 0; i < n; ++i) {
                        const uint32_t j = issued - 1u - i;
                        if (!wait_drain(full0 + 8 * (j % uint32_t(S)), (j / uint32_t(S)) & 1u, p.timeout_ns))
                            atomicOr(p.watchdog, 1u | (1u << (7u + kSiteProducerDrain)));
                    }
                } else {
                    spin_ns(200000);   // this CTA's bytes complete on the first CTA's barrier
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop, so that the stage counters and the
        // descriptors stay warp-uniform, and one elected lane issues.  (Run by
        // lane 0 alone, with descriptors recomputed from kb % S, the same loop
        // measured about 456 instead of 240 cycles per 64-k block at N = 32 or
        // 64; the tensor pipe needs 64 or 128.)
        if (prank == 0) {
            const uint32_t leader = ptx::elect_one();
            const uint64_t ad0 = sdesc_sw128(sA), bd0 = sdesc_sw128(sB);
            uint32_t s = 0, ph = 0;
            bool ok = true;
            for (uint32_t i = 0; i < nkb; ++i) {
                const bool got = wait(full0 + 8 * s, ph, w, kSiteMmaFull);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // stage s: its A and B tiles start s·kABytes and s·kBBytes further (16-byte units)
                const uint64_t ad = ad0 + uint64_t(s * uint32_t(Cfg::kABytes >> 4));
                const uint64_t bd = bd0 + uint64_t(s * uint32_t(Cfg::kBBytes >> 4));
                if (leader) {
#pragma unroll
                    for (int k = 0; k < kBlockK / kUmmaK; ++k)   // 16 k = 32 bytes along the row: +2
                        ptx::mma_f16<CG>(tmem_base, ad + 2u * uint32_t(k), bd + 2u * uint32_t(k), Cfg::kIdesc,
                                         (i != 0 || k != 0) ? 1u : 0u);
                    if constexpr (CG == 2) ptx::mma_commit_pair(empty0 + 8 * s, 0x3);
                    else ptx::mma_commit(empty0 + 8 * s);
                }
                __syncwarp();
                if (++s == uint32_t(S)) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (leader) {
                if (ok) {
                    if constexpr (CG == 2) ptx::mma_commit_pair(acc_full, 0x3);
                    else ptx::mma_commit(acc_full);
                }
                // Every MMA must have retired before the tensor memory is released.
                if constexpr (CG == 2) ptx::mma_commit_pair(mma_done, 0x1);
                else ptx::mma_commit(mma_done);
                if (!wait_drain(mma_done, 0, p.timeout_ns))
                    atomicOr(p.watchdog, 1u | (1u << (7u + kSiteMmaDrain)));
            }
        }
        __syncwarp();
    }

    // ---------------------------------------------------------------- epilogue
    {
        uint32_t ok = 0;
        if (lane == 0) ok = wait(acc_full, 0, wi, kSiteEpiAccFull) ? 1u : 0u;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        const uint32_t taddr = tmem_base + ((warp * 32u) << 16);   // lanes 32w.. = rows 32w..
        // this warp's partial tile and flag (split-K): [BN/4 column groups][32 rows]
        // float4, so that the 32 lanes (rows) of one access cover 512 contiguous bytes
        const uint32_t slot = (cluster * CG + prank) * 4u + warp;
        constexpr uint32_t kSlotF4 = uint32_t(BN / 4) * 32u;           // float4 per warp partial
        float4* const part = reinterpret_cast<float4*>(p.partials) + size_t(slot) * kSlotF4 + lane;
        // a warp's scratch in the ring (split-K), same layout as its partial slot
        const uint32_t scr = sA + warp * uint32_t(Cfg::kScratchBytes);
        const uint32_t xfer = ptx::smem_u32(&ctl->xfer[warp]);
        if (Cfg::kSplit && ok && piece != 0) {
            // a partial piece: the fp32 partial tile through scratch to the
            // workspace with one bulk copy a warp, then the flag once it is complete
            ptx::tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c0), v);
                ptx::tmem_wait_ld();
                ptx::reg_fence(v);
#pragma unroll
                for (int e = 0; e < 8; ++e)   // float4 group c0/4 + e of this lane's row
                    ptx::st_shared_v4(scr + ((uint32_t(c0 / 4 + e) * 32u + lane) << 4), v[4 * e], v[4 * e + 1],
                                      v[4 * e + 2], v[4 * e + 3]);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::bulk_store(part - lane, scr, uint32_t(Cfg::kPartialBytes));
                ptx::bulk_commit_group();
                ptx::bulk_wait_group_all();           // the partial is in global memory
                ptx::fence_proxy_async_global();
                ptx::st_release_u64(p.flags + slot, p.launch_id);
            }
        } else if (ok) {
            ptx::tc_fence_after();
            // the tile's owner: with split-K, lane i waits for piece i's same warp
            // (all at once), then lane 0 loads their partials into scratch together
            uint32_t okf = 1;
            if constexpr (Cfg::kSplit) {
                if (lane >= 1 && lane < p.pieces)
                    okf = wait_flag(p.flags + slot + lane * uint32_t(CG) * 4u, p.launch_id, wi, kSiteStreamK) ? 1u : 0u;
                okf = __all_sync(0xffffffffu, okf) ? 1u : 0u;
                if (okf && lane == 0) {
                    ptx::fence_proxy_async_global();
                    ptx::mbar_arrive_expect_tx(xfer, (p.pieces - 1) * uint32_t(Cfg::kPartialBytes));
                    for (uint32_t i = 1; i < p.pieces; ++i)
                        ptx::bulk_load(scr + (i - 1) * uint32_t(Cfg::kPartialBytes),
                                       part - lane + size_t(i) * uint32_t(CG) * 4u * kSlotF4,
                                       uint32_t(Cfg::kPartialBytes), xfer);
                }
                if (okf && !wait(xfer, 0, wi, kSiteStreamK)) okf = 0;
                okf = __all_sync(0xffffffffu, okf) ? 1u : 0u;
            }
            const int32_t r = m0 + int32_t(warp * 32u + lane);
            uint16_t* crow = p.C + int64_t(r) * p.ldc;
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 64) {
                if (!okf) break;
                // up to 64 columns in registers per wait
                constexpr int kPer = BN < 64 ? BN : 64;
                uint32_t v[2][32];
                ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c0), v[0]);
                if constexpr (kPer == 64) ptx::tmem_ld_32x32b_x32(taddr + uint32_t(c0 + 32), v[1]);
                ptx::tmem_wait_ld();
                ptx::reg_fence(v[0]);
                if constexpr (kPer == 64) ptx::reg_fence(v[1]);
                // the other pieces' partials, in piece order (k order) after this one
                for (uint32_t i = 1; Cfg::kSplit && i < p.pieces; ++i) {
                    // (plain loads, so that the compiler issues them together)
                    const float4* src = reinterpret_cast<const float4*>(
                        smem_raw + (scr - raw) + (i - 1) * uint32_t(Cfg::kPartialBytes)) + lane;
#pragma unroll
                    for (int h = 0; h < kPer / 32; ++h)
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float4 t = src[(c0 / 4 + h * 8 + e) * 32];
                            v[h][4 * e] = __float_as_uint(__uint_as_float(v[h][4 * e]) + t.x);
                            v[h][4 * e + 1] = __float_as_uint(__uint_as_float(v[h][4 * e + 1]) + t.y);
                            v[h][4 * e + 2] = __float_as_uint(__uint_as_float(v[h][4 * e + 2]) + t.z);
                            v[h][4 * e + 3] = __float_as_uint(__uint_as_float(v[h][4 * e + 3]) + t.w);
                        }
                }
#pragma unroll
                for (int h = 0; h < kPer / 32; ++h) {
                    uint32_t q[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        q[e] = Cfg::kBF ? ptx::pack_bf16x2_rn(v[h][2 * e], v[h][2 * e + 1])
                                        : ptx::pack_f16x2_rn(v[h][2 * e], v[h][2 * e + 1]);
                    if (r < p.M) {
#pragma unroll
                        for (int g = 0; g < 4; ++g) {   // 8 columns = 16 bytes each
                            const int32_t n = n0 + c0 + h * 32 + g * 8;
                            if (n + 8 <= p.N) {
                                *reinterpret_cast<uint4*>(crow + n) =
                                    make_uint4(q[4 * g], q[4 * g + 1], q[4 * g + 2], q[4 * g + 3]);
                            } else {
                                for (int e = 0; e < 8 && n + e < p.N; ++e)
                                    crow[n + e] = uint16_t(q[4 * g + e / 2] >> (16 * (e & 1)));
                            }
                        }
                    }
                }
            }
        }
    }

    ptx::tc_fence_before();
    if constexpr (CG == 2) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
}

}  // namespace g16
