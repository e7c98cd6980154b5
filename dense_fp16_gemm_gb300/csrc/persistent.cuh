// The persistent kernel of the GB300 (sm_103a) dense fp16 NT GEMM library:
// C[M,N] = A[M,K] · B[N,K]ᵀ, fp32 accumulation (an fp16 accumulator and bf16
// operands on request).  Device code only; gemm_f16_nt.cu holds the host side.
//
// One persistent kernel, warp-specialised:
//   warp 0      TMA producer: fills an S-stage shared-memory ring (A tile + B
//               tile per stage, 128-byte swizzled) gated by full/empty mbarriers;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (kind::f16, fp32
//               accumulate) into tensor memory, frees ring slots with
//               tcgen05.commit, and hands finished accumulators to the epilogue;
//   warps 2-5   epilogue: tcgen05.ld → fp32→fp16 round-to-nearest-even →
//               swizzled shared-memory staging → TMA store, clipped at M/N.
// Two TMEM accumulator buffers let the epilogue of one tile overlap the main
// loop of the next.  In the default configuration a cluster of two CTAs runs
// 2-SM MMAs (cta_group::2) on a 256×256 tile: each CTA loads its own 128 rows of
// A and one half of the B tile, and the pair's single MMA reads both halves, so
// the shared operand crosses L2 once per pair.
//
// Variants, all in this one kernel template (KCfg): one CTA per tile
// (cta_group::1); bf16 operands and result; an fp16 accumulator; A and/or B
// stored M/N-contiguous (MN-major operands); and, only in the separately built
// single-GPU library (mcast/gemm_f16_nt_mcast.cu, which includes gemm_f16_nt.cu), a
// cluster of two pairs that share A by TMA multicast.  The work schedule (see "work schedule") mixes whole tiles, a
// stream-K split of the last wave in k, and column slices of small problems'
// tiles.  Launches use programmatic dependent launch: a CTA sets up, then
// waits for the previous kernel on the stream before touching global memory.
//
// Design lineage (prior art, re-derived for tcgen05): the Tilus matmul-hopper
// tutorial's V2 ring buffer ("2. Multi-Stage Software Pipelining"), V3 role
// split and full/empty barriers ("3. Warp Specialization", §Producer-Consumer
// Barriers), V4 raster ("4. Pipeline Abstraction and Two Consumer Warp Groups",
// §Tile Rasterization) and V6 cluster pairing, persistent loop and TMA-store
// epilogue ("6. Register Reallocation, Multicast, and a Persistent Kernel",
// §Cluster Multicast, §Persistent Tile Loop, §Shared-Memory Epilogue).  The
// accumulator lives in TMEM instead of registers, so V6's register
// reallocation (§The Register Budget Problem) has no counterpart here.
//
// Every wait on an mbarrier or a flag is bounded by a watchdog: a wait for one
// pipeline stage by the base limit (default 1 s), a wait that can span a whole
// work item's main loop by the base limit plus a fixed allowance per k-block of
// a tile.  On expiry the CTA sets a flag that ends every role's loop, records
// the expired wait in a device word, waits (bounded) for its own copies and MMAs
// in flight, releases its tensor memory and exits.

#pragma once

#include <cuda.h>
#include <stdint.h>

#include <type_traits>

#include "ptx.cuh"
#include "sched.cuh"

// 1 when this header is compiled into the single-GPU multicast library (whose
// translation unit defines it and provides McastA first); 0 in the default
// library, which has no multicast load.
#ifndef G16_MCAST_LIB
#define G16_MCAST_LIB 0
#endif

namespace g16 {

#if !G16_MCAST_LIB
// The default library has no loader for clusters of two pairs.
template <int CP>
struct McastA {
    static constexpr bool kAvailable = false;
};
#endif

constexpr int kBlockM = 128;   // accumulator rows per CTA = TMEM lanes
constexpr int kBlockK = 64;    // k per stage: 64 fp16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;     // k per tcgen05.mma of kind::f16
constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kEpiWarps = 4;
constexpr int kEpiCols = 64;                       // columns per staged store (128-byte rows)
constexpr int kOutBufBytes = 32 * kEpiCols * 2;    // one warp's 32×64 fp16 staging tile
constexpr int kOutBufs = 2;                        // double-buffered per warp
constexpr int kDefaultSwizzle = 8;
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;
// Allowance per k-block of a tile for the waits that can span a work item's
// whole main loop (a k-block takes about 0.27 us at full clock; 8 us leaves a
// margin of about 30x for low clocks and contention).
constexpr uint64_t kItemWaitNsPerKb = 8000ull;

// watchdog word layout: bit 0 = a wait expired, bit 7+s = wait site s expired
enum : uint32_t {
    kSiteProducerEmpty = 1,
    kSiteMmaFull = 2,
    kSiteMmaAccFree = 3,
    kSiteEpiAccFull = 4,
    kSiteProducerDrain = 5,
    kSiteMmaDrain = 6,
    kSiteStreamK = 7,
    kSiteClaim = 8,
};

__device__ uint32_t g_watchdog_word;

// Counters of the last-wave claims (Params::claim): a launch takes the word
// of its id modulo kClaimWords, so that launches running at the same time on
// other streams use other words (each word is tagged with its last launch).
constexpr int kClaimWords = 256;
__device__ unsigned long long g_claim_words[kClaimWords];

template <int CG, int BN, int STAGES, int CP = 1, bool BF = false, bool A16 = false>
struct KCfg {
    static constexpr int kCG = CG;
    static constexpr bool kBF = BF;                  // bf16 operands and result instead of fp16
    static constexpr bool kA16 = A16;                // fp16 accumulator instead of fp32
    static constexpr int kCP = CP;                   // CTA pairs per cluster (A shared by multicast)
    static constexpr int kCtas = CG * CP;            // CTAs per cluster
    static constexpr int kBN = BN;                   // columns of C per tile
    static constexpr int kStages = STAGES;
    static constexpr int kTileM = kBlockM * CG;      // rows of C per tile
    static constexpr int kBRows = BN / CG;           // B rows this CTA loads per stage
    static constexpr int kABytes = kBlockM * kBlockK * 2;
    static constexpr int kBBytes = kBRows * kBlockK * 2;
    static constexpr int kTxBytes = (kABytes + kBBytes) * CG;  // bytes per stage on the leader's barrier
    static constexpr int kTmemCols = 2 * BN <= 32 ? 32 : 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128
                                   : 2 * BN <= 256 ? 256 : 512;
    static constexpr int kRingBytes = STAGES * (kABytes + kBBytes);
    static constexpr int kOutBytes = kEpiWarps * kOutBufs * kOutBufBytes;
    static constexpr int kCtlBytes = 256;
    static constexpr int kSmemBytes = 1024 + kRingBytes + kOutBytes + kCtlBytes;
    // tcgen05 instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1) or fp16
    // (= 0), A and B fp16 (bits 7-9, 10-12 = 0) or bf16 (= 1), both K-major
    // (bits 15, 16 = 0), N>>3 at bit 17, M>>4 at bit 24.  An fp16 D takes the
    // same TMEM columns as fp32: one value per 32-bit column, in its low half.
    static constexpr uint32_t kIdesc = (uint32_t(!A16) << 4) | (uint32_t(BF) << 7) | (uint32_t(BF) << 10) |
                                       (uint32_t(BN >> 3) << 17) | (uint32_t(kTileM >> 4) << 24);

    static_assert(2 * BN <= 512, "two accumulator buffers must fit in the 512 TMEM columns");
    static_assert(BN % kEpiCols == 0, "epilogue works in 64-column chunks");
    static_assert(kBRows <= 256, "a TMA box is at most 256 rows");
    static_assert(kSmemBytes <= 232448, "dynamic shared memory limit per CTA");
    static_assert(CP == 1 || (CG == 2 && CP == 2), "two pairs per cluster only with CTA pairs");
    static_assert(!(A16 && BF), "an fp16 accumulator needs fp16 operands");
};

template <int STAGES>
struct Ctl {
    uint64_t full[STAGES];      // stage loaded (TMA bytes landed)   — leader CTA's copy is used
    uint64_t empty[STAGES];     // stage consumed (MMAs done)        — each CTA's own copy
    uint64_t acc_full[2];       // accumulator ready for the epilogue
    uint64_t acc_empty[2];      // accumulator drained               — leader CTA's copy is used
    uint64_t mma_done;          // all MMAs retired (teardown)
    uint64_t xfer[kEpiWarps];   // split pieces: partial slices landed in an epilogue warp's scratch
    uint64_t claim_bar;         // the cluster's claim of a last-wave tile is in claim_tile
    uint32_t claim_tile;
    uint32_t tmem_base;
    uint32_t abort_flag;
};

struct Params {
    CUtensorMap tmA;   // A: dims {K, M}, box {64, 128}
    CUtensorMap tmB;   // B: dims {K, N}, box {64, BN/CG}
    CUtensorMap tmBp;  // B for N-split tail tiles: box {64, BN/CG/tail_split}
    CUtensorMap tmC;   // C: dims {N8, M}, box {64, 32}; only when N8 > 0
    Raster raster;
    uint32_t num_tiles;
    uint32_t num_kb;
    int32_t M;
    int32_t N;
    int32_t N8;        // N rounded down to a multiple of 8 (16 bytes)
    uint16_t* C;       // for the last N - N8 columns, written with plain stores
    int64_t ldc;
    uint64_t timeout_ns;       // limit of a wait for one pipeline stage
    uint64_t item_timeout_ns;  // limit of a wait that can span a work item's main loop
    uint32_t* watchdog;
    int32_t inject_stall;
    uint32_t a_mn;     // 1: A stored [K, M] (M contiguous) — MN-major in shared memory
    uint32_t b_mn;     // 1: B stored [K, N] (N contiguous)
    // stream-K part of the schedule (0 tiles = purely data-parallel)
    uint32_t sk_tiles;     // tiles [0, sk_tiles) are cut into k-block units
    uint64_t sk_units;     // sk_tiles * num_kb
    float* partials;       // [cluster][cta rank][BN/4][128 rows] float4 partial tiles
    uint64_t* flags;       // [cluster][cta rank][epilogue warp]: launch_id once written
    uint64_t launch_id;    // unique per launch, so stale flags never match
    // N-split tail: tiles [tail_first, num_tiles) are each cut into tail_split
    // tiles of BN/tail_split columns (tail_first = num_tiles: no split)
    uint32_t tail_first;
    uint32_t tail_split;
    uint32_t split_pieces; // > 1: each cluster runs one split piece of tile cluster / split_pieces
    uint32_t k_alternate;  // 1: whole tiles of odd rounds load k from the top down (item_k_down)
    // Whole tiles [dyn_first, num_tiles) (a last, partial wave) are claimed at
    // run time, one at most per cluster, through the 64-bit word *claim: the
    // launch's tag (the low 32 bits of launch_id) above a 32-bit count of
    // tickets taken.
    uint32_t dyn_first;
    unsigned long long* claim;
    uint64_t* trace;       // optional per-item timestamps (debugging)
    uint32_t trace_items;
};

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------

struct Watch {
    uint64_t limit_ns;
    volatile uint32_t* abort_flag;   // this CTA's flag
    uint32_t abort_addr;             // its shared-memory address (same offset in every CTA)
    uint32_t ctas;                   // CTAs in the cluster
    uint32_t rank;                   // this CTA's rank in the cluster
    uint32_t* word;
};

// Stop this CTA and every other CTA of the cluster (they wait on each other).
__device__ __noinline__ void raise_abort(const Watch w, uint32_t site) {
    *w.abort_flag = 1u;
    for (uint32_t r = 0; r < w.ctas; ++r)
        if (r != w.rank) ptx::st_cluster_u32(ptx::mapa(w.abort_addr, r), 1u);
    atomicOr(w.word, 1u | (1u << (7u + site)));
}

// A ticket for the last-wave tiles of the launch tagged `launch_id`.  The
// 64-bit word holds the tag (the low 32 bits of the id) of the launch that
// started its count above the count of tickets taken (32 bits).  Cluster 0
// starts the count at the launch's start (claim_start); a claim is one atomic
// add (the clusters claim at about the same time, and a contended
// compare-and-swap loop costs microseconds of retries there).  An add that
// finds an older launch's tag came before the start: the start overwrites its
// increment, and the claimer waits for the new tag and adds again.  Returns
// the ticket, or kNoTicket if the tag did not come within `limit_ns`.
constexpr uint32_t kNoTicket = 0xFFFFFFFFu;
__device__ __forceinline__ void claim_start(unsigned long long* w, uint64_t launch_id) {
    atomicExch(w, (launch_id & 0xFFFFFFFFull) << 32);
}
__device__ __noinline__ uint32_t claim_ticket(unsigned long long* w, uint64_t launch_id, uint64_t limit_ns) {
    const unsigned long long tag = launch_id & 0xFFFFFFFFull;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        const unsigned long long v = atomicAdd(w, 1ull);
        if ((v >> 32) == tag) return uint32_t(v & 0xFFFFFFFFull);
        while ((atomicAdd(w, 0ull) >> 32) != tag) {
            if (ptx::globaltimer() - t0 > limit_ns) return kNoTicket;
            __nanosleep(256);
        }
    }
}

// Between checks of the watchdog, a waiting thread sleeps in the barrier
// (woken when the phase completes) rather than polling shared memory, which
// would take issue slots and shared-memory bandwidth from the tensor cores.
constexpr uint32_t kWaitSleepNs = 20000;

// (kCluster: the wait acquires at cluster scope, for a barrier that a thread
// of another CTA arrives on after writing what the waiter then reads.)
template <bool kCluster = false>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Watch w, uint32_t site) {
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        if (kCluster ? ptx::mbar_try_wait_sleep_acq_cluster(bar, parity, kWaitSleepNs)
                     : ptx::mbar_try_wait_sleep(bar, parity, kWaitSleepNs))
            return true;
        if (*w.abort_flag) return false;
        if (ptx::globaltimer() - t0 > w.limit_ns) {
            raise_abort(w, site);
            return false;
        }
    }
}

// Wait for the phase of parity `parity` to complete; false if the watchdog
// fired (here or elsewhere in the CTA).
template <bool kCluster = false>
__device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, const Watch& w, uint32_t site) {
    if (kCluster ? ptx::mbar_try_wait_acq_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow<kCluster>(bar, parity, w, site);
}

// Teardown wait after an abort: ignores the abort flag, bounded by the limit.
__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        if (ptx::mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
        if (ptx::globaltimer() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < ns) {
    }
}

// Shared-memory matrix descriptor for a K-major tile written by TMA with
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked
// along M/N.  Start address >> 4 in bits 0-13, leading-byte offset (unused for
// swizzled K-major) in 16-29, stride-byte offset 1024 >> 4 in 32-45, descriptor
// version 1 in bits 46-47, swizzle mode 2 (128 B) in bits 61-63.  Advancing K by
// 16 fp16 inside the 128-byte row adds 32 bytes (2 in the start field).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// The same for an MN-major tile (M or N contiguous): TMA writes it as 64×64
// boxes, each 64 K-rows of 128 bytes (64 consecutive M/N elements), swizzled in
// 8-row (1024-byte) atoms; the boxes for successive 64-element M/N blocks follow
// each other every 8 KiB.  Leading-byte offset = that 8 KiB step between atoms
// along M/N, stride-byte offset = 1024 bytes between 8-row groups along K.
// Advancing K by 16 moves 16 rows: 2048 bytes.
constexpr uint32_t kMnBoxBytes = 64 * 64 * 2;
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr) {
    return uint64_t((saddr & 0x3FFFFu) >> 4) | (uint64_t(kMnBoxBytes >> 4) << 16) |
           (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Wait until *flag == want (the partner's release store); false on watchdog.
__device__ __noinline__ bool wait_flag(const uint64_t* flag, uint64_t want, const Watch w,
                                       uint32_t site) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (ptx::ld_acquire_u64(flag) == want) return true;
        if ((i & 15u) == 0) {
            if (*w.abort_flag) return false;
            if (ptx::globaltimer() - t0 > w.limit_ns) {
                raise_abort(w, site);
                return false;
            }
        }
        __nanosleep(64);
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <class Cfg>
__global__ void __launch_bounds__(kThreads, 1) gemm_f16_nt_kernel(const __grid_constant__ Params p) {
    constexpr int CG = Cfg::kCG;
    constexpr int CP = Cfg::kCP;
    constexpr int NCTA = Cfg::kCtas;
    constexpr int BN = Cfg::kBN;
    constexpr int S = Cfg::kStages;
    static_assert(CP == 1 || McastA<CP>::kAvailable, "two pairs per cluster need the multicast library's loader");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // 128-byte swizzle atoms need 1 KB alignment
    const uint32_t sA = base;
    const uint32_t sB = sA + S * Cfg::kABytes;
    const uint32_t sOut = sB + S * Cfg::kBBytes;
    Ctl<S>* ctl = reinterpret_cast<Ctl<S>*>(smem_raw + (base - raw) + Cfg::kRingBytes + Cfg::kOutBytes);

    const uint32_t warp = __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t rank = NCTA > 1 ? ptx::cluster_ctarank() : 0u;   // rank in the cluster
    const uint32_t pair = CG == 2 ? rank >> 1 : 0u;                  // CTA pair in the cluster
    const uint32_t prank = CG == 2 ? rank & 1u : 0u;                 // rank in the pair
    const uint32_t lead = pair * 2u;                                 // the pair's leader CTA
    const uint32_t cluster = NCTA > 1 ? ptx::cluster_id_x() : blockIdx.x;
    const uint32_t nclusters = NCTA > 1 ? ptx::nclusters_x() : gridDim.x;

    const uint32_t full0 = ptx::smem_u32(&ctl->full[0]);
    const uint32_t empty0 = ptx::smem_u32(&ctl->empty[0]);
    const uint32_t accf0 = ptx::smem_u32(&ctl->acc_full[0]);
    const uint32_t acce0 = ptx::smem_u32(&ctl->acc_empty[0]);
    const uint32_t mma_done = ptx::smem_u32(&ctl->mma_done);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);     // the leader's expect-tx arrive
            ptx::mbar_init(empty0 + 8 * s, CP);   // one tcgen05.commit from each pair's leader
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(accf0 + 8 * b, 1);                  // one tcgen05.commit
            ptx::mbar_init(acce0 + 8 * b, kEpiWarps * CG);     // every epilogue warp of the pair
        }
        ptx::mbar_init(mma_done, 1);
        for (int e = 0; e < kEpiWarps; ++e) ptx::mbar_init(ptx::smem_u32(&ctl->xfer[e]), 1);
        ptx::mbar_init(ptx::smem_u32(&ctl->claim_bar), 1);   // the claiming producer's arrive
        ctl->abort_flag = 0u;
        ptx::fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&p.tmA);
        ptx::prefetch_tensormap(&p.tmB);
        if (p.N8 > 0) ptx::prefetch_tensormap(&p.tmC);
    }
    if (warp == 1) {
        ptx::tmem_alloc<CG>(ptx::smem_u32(&ctl->tmem_base), Cfg::kTmemCols);
        ptx::tmem_relinquish<CG>();
    }
    ptx::tc_fence_before();
    if constexpr (NCTA > 1) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(&ctl->tmem_base);

    // Programmatic dependent launch: the next kernel on the stream may start
    // its own set-up as soon as SMs free up; everything above touched only this
    // CTA's shared and tensor memory.  Global memory (operands, C, workspace,
    // watchdog word) is touched only after the previous kernel on the stream has
    // completed and its writes are visible.
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();
    // this launch's count of claimed tiles starts at 0 (claim_ticket)
    if (p.dyn_first < p.num_tiles && cluster == 0 && rank == 0 && threadIdx.x == 0) claim_start(p.claim, p.launch_id);

    Watch w;
    w.limit_ns = p.timeout_ns;
    w.abort_flag = &ctl->abort_flag;
    w.abort_addr = ptx::smem_u32(&ctl->abort_flag);
    w.ctas = NCTA;
    w.rank = rank;
    w.word = p.watchdog;
    // Waits that can legitimately last a whole work item: the epilogue's wait
    // for a finished accumulator, an owner's wait for its partners' partial
    // tiles, the MMA issuer's wait for a drained accumulator and, behind it, the
    // producer's wait for a free stage.  Only the MMA issuer's wait for a filled
    // stage (which depends on nothing but the copies in flight) keeps the base
    // limit.
    Watch wi = w;
    wi.limit_ns = p.item_timeout_ns;

    // The last wave's tiles (work_next's `claim`).  The cluster's first
    // producer (rank 0), once it has issued its share of loads, takes a ticket
    // and publishes the tile it names (or num_tiles: none) to every CTA of the
    // cluster; every other role of every CTA reads it there.  So the clusters
    // that finish their share first run the last wave, whatever the speed of
    // their SMs.
    const uint32_t claim_bar = ptx::smem_u32(&ctl->claim_bar);
    auto claim_take = [&]() -> uint32_t {
        uint32_t tile = p.num_tiles;
        const uint32_t ticket = claim_ticket(p.claim, p.launch_id, wi.limit_ns);
        if (ticket == kNoTicket)
            atomicOr(p.watchdog, 1u | (1u << (7u + kSiteClaim)));   // a tile left undone: report it
        else if (ticket < p.num_tiles - p.dyn_first)
            tile = p.dyn_first + ticket;
        if constexpr (NCTA > 1) {
            const uint32_t slot = ptx::smem_u32(&ctl->claim_tile);
            for (uint32_t r = 0; r < uint32_t(NCTA); ++r) {
                ptx::st_cluster_u32(ptx::mapa(slot, r), tile);
                ptx::mbar_arrive_cluster(ptx::mapa(claim_bar, r));
            }
        } else {
            *reinterpret_cast<volatile uint32_t*>(&ctl->claim_tile) = tile;
            ptx::mbar_arrive(claim_bar);
        }
        return tile;
    };
    auto claim_read = [&]() -> uint32_t {
        if (!wait<(NCTA > 1)>(claim_bar, 0, wi, kSiteClaim)) return p.num_tiles;
        return *reinterpret_cast<volatile uint32_t*>(&ctl->claim_tile);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && !p.inject_stall) {
            // Completion bytes of both CTAs' loads go to the pair leader's full barrier.
            const uint32_t full_tgt = CG == 2 ? ptx::mapa(full0, lead) : full0;
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = true;
            // Tiles of one raster group share B column strips across successive
            // waves: keep B in L2 in preference to the streamed A rows.
            const uint64_t keep_b = ptx::policy_evict_last();
            Work work;
            Item it;
            work_init(work, p, cluster, nclusters);
            while (ok && work_next(work, p, it, [&] { return rank == 0 ? claim_take() : claim_read(); })) {
                uint32_t mt, nt;
                raster_coord(p.raster, it.tile, mt, nt);
                const int32_t m0 = int32_t(mt * Cfg::kTileM + prank * kBlockM);
                // an N-split tail item loads BRows/parts rows of B at its column slice
                const int32_t brows = Cfg::kBRows / int32_t(it.parts);
                const int32_t n0 = int32_t((nt * CP + pair) * BN + it.part * (BN / it.parts)) + prank * brows;
                const uint32_t tx = it.parts == 1 ? uint32_t(Cfg::kTxBytes)
                                                  : uint32_t(Cfg::kABytes + Cfg::kBBytes / int32_t(it.parts)) * CG;
                // The k-block order (item_k_down): a partial piece, and a whole
                // tile in an odd round, load from the last k-block down.  The MMA
                // issuer consumes stages in ring order and needs no change.  An
                // fp16 accumulator keeps k order: its rounding depends on it.
                const bool down = !Cfg::kA16 && item_k_down(p, it, nclusters);
                for (uint32_t i = it.kb0; i < it.kb1; ++i) {
                    const uint32_t kb = down ? it.kb1 - 1u - (i - it.kb0) : i;
                    if (!wait(empty0 + 8 * stage, phase ^ 1u, wi, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    if (prank == 0) ptx::mbar_arrive_expect_tx(full0 + 8 * stage, tx);
                    const int32_t k0 = int32_t(kb * kBlockK);
                    const uint32_t bar = full_tgt + 8 * stage;
                    // A K-major operand is one box {64 k, rows}; an MN-major one is
                    // rows/64 boxes {64 m|n, 64 k}, 8 KiB apart, at coordinates (m|n, k).
                    const uint32_t a_dst = sA + stage * Cfg::kABytes;
                    const uint32_t b_dst = sB + stage * Cfg::kBBytes;
                    if constexpr (CP == 2) {
                        // Both pairs need the same A rows: this CTA loads half of them
                        // into the same-rank CTA of both pairs (TMA multicast; the
                        // loader exists only in the single-GPU multicast library).
                        const int32_t r0 = m0 + int32_t(pair * (kBlockM / 2));
                        const uint16_t mask = uint16_t((1u << prank) | (1u << (prank + 2u)));
                        if (p.a_mn)
                            McastA<CP>::load(a_dst + pair * kMnBoxBytes, &p.tmA, r0, k0, bar, mask);
                        else
                            McastA<CP>::load(a_dst + pair * (Cfg::kABytes / 2), &p.tmA, k0, r0, bar, mask);
                    } else if (p.a_mn) {
                        for (int j = 0; j < kBlockM / 64; ++j) {
                            if constexpr (CG == 2)
                                ptx::tma_load_2d_pair(a_dst + j * kMnBoxBytes, &p.tmA, m0 + 64 * j, k0, bar);
                            else
                                ptx::tma_load_2d(a_dst + j * kMnBoxBytes, &p.tmA, m0 + 64 * j, k0, bar);
                        }
                    } else {
                        if constexpr (CG == 2) ptx::tma_load_2d_pair(a_dst, &p.tmA, k0, m0, bar);
                        else ptx::tma_load_2d(a_dst, &p.tmA, k0, m0, bar);
                    }
                    if (p.b_mn) {
                        for (int j = 0; j < Cfg::kBRows / 64; ++j) {
                            if constexpr (CG == 2)
                                ptx::tma_load_2d_pair_hint(b_dst + j * kMnBoxBytes, &p.tmB, n0 + 64 * j, k0, bar, keep_b);
                            else
                                ptx::tma_load_2d_hint(b_dst + j * kMnBoxBytes, &p.tmB, n0 + 64 * j, k0, bar, keep_b);
                        }
                    } else {
                        // (tail items exist only for K-major B with one pair per cluster)
                        const CUtensorMap* mb = it.parts == 1 ? &p.tmB : &p.tmBp;
                        if constexpr (CG == 2) ptx::tma_load_2d_pair_hint(b_dst, mb, k0, n0, bar, keep_b);
                        else ptx::tma_load_2d_hint(b_dst, mb, k0, n0, bar, keep_b);
                    }
                    ++issued;
                    if (++stage == uint32_t(S)) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && issued) {
                // Let the copies already issued land before the CTA can exit.
                if (prank == 0) {
                    uint32_t s = stage, ph = phase;
                    const uint32_t n = issued < uint32_t(S) ? issued : uint32_t(S);
                    for (uint32_t i = 0; i < n; ++i) {
                        if (s == 0) {
                            s = S - 1;
                            ph ^= 1u;
                        } else {
                            --s;
                        }
                        if (!wait_drain(full0 + 8 * s, ph, p.timeout_ns))
                            atomicOr(p.watchdog, 1u | (1u << (7u + kSiteProducerDrain)));
                    }
                } else {
                    spin_ns(200000);   // this CTA's bytes complete on the peer's barrier
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && prank == 0) {
            // One thread issues every MMA of the pair, and a few extra instructions
            // per k-block are enough to leave the tensor pipe idle between stages:
            // the loop is compiled once per operand layout, so that inside it a
            // stage and a 16-k step only move the descriptors' start-address field
            // by compile-time amounts (16-byte units).
            auto issue = [&](auto a_mn_tag, auto b_mn_tag) {
                constexpr bool kAmn = decltype(a_mn_tag)::value;
                constexpr bool kBmn = decltype(b_mn_tag)::value;
                // bits 15 / 16: A / B MN-major ("transposed") in shared memory
                constexpr uint32_t idesc = Cfg::kIdesc | (uint32_t(kAmn) << 15) | (uint32_t(kBmn) << 16);
                // per 16-k step: 32 bytes along a K-major row, 16 rows (2048 bytes) MN-major
                constexpr uint32_t a_kstep = kAmn ? (kUmmaK * 128) >> 4 : (kUmmaK * 2) >> 4;
                constexpr uint32_t b_kstep = kBmn ? (kUmmaK * 128) >> 4 : (kUmmaK * 2) >> 4;
                uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
                bool ok = true;
                Work work;
                Item it;
                work_init(work, p, cluster, nclusters);
                uint32_t item_no = 0;
                while (ok && work_next(work, p, it, claim_read)) {
                    if (!wait(acce0 + 8 * acc, acc_phase ^ 1u, wi, kSiteMmaAccFree)) break;
                    ptx::tc_fence_after();
                    uint64_t* tr = (p.trace && item_no < p.trace_items)
                                       ? p.trace + (size_t(cluster) * p.trace_items + item_no) * 8 : nullptr;
                    if (tr) {
                        tr[0] = uint64_t(it.tile) | (uint64_t(it.kind) << 32);
                        tr[1] = uint64_t(it.kb0) | (uint64_t(it.kb1) << 32);
                        tr[2] = ptx::globaltimer();
                    }
                    ++item_no;
                    const uint32_t d = tmem_base + acc * uint32_t(BN);
                    uint64_t starved_ns = 0;   // traced: time spent waiting for filled stages
                    // The k-block loop, compiled once per MMA width so that the
                    // instruction descriptor stays a compile-time constant (a
                    // descriptor in a register slows the issuing thread by ~2 %).
                    auto kloop = [&](auto id_tag) {
                        constexpr uint32_t id = decltype(id_tag)::value;
                        for (uint32_t kb = it.kb0; kb < it.kb1; ++kb) {
                            if (tr && !ptx::mbar_test_wait(full0 + 8 * stage, phase)) {
                                const uint64_t ts = ptx::globaltimer();
                                ok = wait(full0 + 8 * stage, phase, w, kSiteMmaFull);
                                starved_ns += ptx::globaltimer() - ts;
                            } else if (!tr) {
                                ok = wait(full0 + 8 * stage, phase, w, kSiteMmaFull);
                            }
                            if (!ok) break;
                            ptx::tc_fence_after();
                            const uint32_t sa = sA + stage * uint32_t(Cfg::kABytes);
                            const uint32_t sb = sB + stage * uint32_t(Cfg::kBBytes);
                            const uint64_t ad = kAmn ? sdesc_sw128_mn(sa) : sdesc_sw128(sa);
                            const uint64_t bd = kBmn ? sdesc_sw128_mn(sb) : sdesc_sw128(sb);
#pragma unroll
                            for (int k = 0; k < kBlockK / kUmmaK; ++k) {
                                ptx::mma_f16<CG>(d, ad + a_kstep * uint32_t(k), bd + b_kstep * uint32_t(k), id,
                                                 (kb != it.kb0 || k != 0) ? 1u : 0u);
                            }
                            // Free this ring slot in every CTA of the pair once these MMAs retire.
                            // (with two pairs, the stage is free only once both pairs' MMAs are done)
                            if constexpr (CG == 2) ptx::mma_commit_pair(empty0 + 8 * stage, CP == 2 ? 0xF : 0x3);
                            else ptx::mma_commit(empty0 + 8 * stage);
                            if (++stage == uint32_t(S)) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    };
                    // an N-split item's MMAs are BN/parts wide (descriptor N>>3 at bit 17)
                    constexpr uint32_t kNoN = idesc & ~(0x3Fu << 17);
                    if (it.parts == 1)
                        kloop(std::integral_constant<uint32_t, idesc>{});
                    else if (it.parts == 2)
                        kloop(std::integral_constant<uint32_t, kNoN | (uint32_t(BN / 2 / 8) << 17)>{});
                    else
                        kloop(std::integral_constant<uint32_t, kNoN | (uint32_t(BN / 4 / 8) << 17)>{});
                    if (!ok) break;
                    if constexpr (CG == 2) ptx::mma_commit_pair(accf0 + 8 * acc, uint16_t(0x3u << lead));
                    else ptx::mma_commit(accf0 + 8 * acc);
                    if (tr) {
                        tr[3] = ptx::globaltimer();
                        tr[7] = starved_ns;
                    }
                    acc ^= 1u;
                    if (acc == 0) acc_phase ^= 1u;
                }
            };
            using K_ = std::false_type;
            using T_ = std::true_type;
            if (p.a_mn) {
                if (p.b_mn) issue(T_{}, T_{});
                else issue(T_{}, K_{});
            } else {
                if (p.b_mn) issue(K_{}, T_{});
                else issue(K_{}, K_{});
            }
            // Every MMA must have retired before the tensor memory is released.
            if constexpr (CG == 2) ptx::mma_commit_pair(mma_done, uint16_t(1u << lead));
            else ptx::mma_commit(mma_done);
            if (!wait_drain(mma_done, 0, p.timeout_ns)) atomicOr(p.watchdog, 1u | (1u << (7u + kSiteMmaDrain)));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const uint32_t q = warp & 3u;                      // TMEM lane quarter this warp may read
        const uint32_t lane_off = (q * 32u) << 16;
        const uint32_t out0 = sOut + (warp - 2u) * kOutBufs * kOutBufBytes;
        const uint32_t acce_tgt = CG == 2 ? ptx::mapa(acce0, lead) : acce0;
        // A partial tile in workspace slot `slot` is stored as float4 groups of
        // columns, row innermost: [col/4][128 rows], so that the 32 lanes of a
        // warp (32 consecutive rows) touch 512 contiguous bytes per access.
        // Layout [slot][cta rank][epilogue warp][BN/4 column groups][32 rows]:
        // a warp's partial rows are contiguous, 8 KB per 64 columns, and the 32
        // lanes (rows) of one float4 column group touch 512 contiguous bytes.
        auto partial_f4 = [&](uint32_t slot, uint32_t col4) {
            return reinterpret_cast<float4*>(p.partials) +
                   (((size_t(slot) * NCTA + rank) * kEpiWarps + q) * (BN / 4) + col4) * 32u + lane;
        };
        uint32_t acc = 0, acc_phase = 0, ob = 0;
        Work work;
        Item it;
        work_init(work, p, cluster, nclusters);
        uint32_t item_no = 0;
        while (work_next(work, p, it, claim_read)) {
            uint32_t mt, nt;
            raster_coord(p.raster, it.tile, mt, nt);
            const int32_t row0 = int32_t(mt * Cfg::kTileM + prank * kBlockM + q * 32u);
            const int32_t col0 = int32_t((nt * CP + pair) * BN + it.part * (BN / it.parts));
            const int nchunks = (BN / kEpiCols) / int(it.parts);
            uint64_t* tr = (p.trace && item_no < p.trace_items && rank == 0 && warp == 2 && lane == 0)
                               ? p.trace + (size_t(cluster) * p.trace_items + item_no) * 8 : nullptr;
            ++item_no;
            uint32_t ok = 0;
            if (lane == 0) ok = wait(accf0 + 8 * acc, acc_phase, wi, kSiteEpiAccFull) ? 1u : 0u;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ptx::tc_fence_after();
            if (tr) tr[4] = ptx::globaltimer();
            if constexpr (!Cfg::kA16) {
                if (it.kind == kItemSplitPiece) {
                    // One of `np` split pieces of the tile, all running at once on
                    // clusters first .. first+np-1.  The tile's BN columns are cut
                    // into np contiguous slices, piece i owning slice i.  The
                    // pieces exchange partials through the workspace with bulk
                    // copies, staged in this warp's share of the ring (idle now:
                    // a split piece is its cluster's only item, and its last
                    // stage was consumed before the accumulator was ready):
                    //  1. the fp32 partials of the slices other pieces own are
                    //     written to scratch and stored to this cluster's slot;
                    //  2. once they are complete, a release flag publishes them;
                    //  3. after the same warp of every other piece has published,
                    //     their partials of this piece's slice are loaded back
                    //     together, summed with its own in piece order (k order)
                    //     and stored to C.
                    const uint32_t np = it.pieces, pc = it.piece, first = cluster - pc;
                    const uint32_t tacc = tmem_base + lane_off + acc * uint32_t(BN);
                    const uint32_t own0 = pc * (BN / 32) / np, own1 = (pc + 1) * (BN / 32) / np;  // 32-col slices
                    constexpr uint32_t kScratch = Cfg::kRingBytes / kEpiWarps;
                    static_assert(kScratch >= 7 * 4096 && kScratch >= (BN / 32) * 4096, "split-piece scratch");
                    const uint32_t scr = sA + q * kScratch;    // ring is [sA, sA + kRingBytes)
                    // 1. partial slices for the other pieces, 4 KB each: [8 column groups][32 rows] float4
                    uint32_t nst = 0;
#pragma unroll 1
                    for (uint32_t c = 0; c < uint32_t(BN / 64); ++c) {
                        const bool own_lo = 2 * c >= own0 && 2 * c < own1;
                        const bool own_hi = 2 * c + 1 >= own0 && 2 * c + 1 < own1;
                        if (own_lo && own_hi) continue;
                        uint32_t lo[32], hi[32];
                        ptx::tmem_ld_32x32b_x32(tacc + 64 * c, lo);
                        ptx::tmem_ld_32x32b_x32(tacc + 64 * c + 32, hi);
                        ptx::tmem_wait_ld();
                        ptx::reg_fence(lo);
                        ptx::reg_fence(hi);
                        const uint32_t blk = scr + 8192u * c;    // scratch mirrors the slot's layout
                        if (!own_lo)
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                ptx::st_shared_v4(blk + (uint32_t(k) * 32u + lane) * 16u, lo[4 * k], lo[4 * k + 1],
                                                  lo[4 * k + 2], lo[4 * k + 3]);
                        if (!own_hi)
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                ptx::st_shared_v4(blk + 4096u + (uint32_t(k) * 32u + lane) * 16u, hi[4 * k],
                                                  hi[4 * k + 1], hi[4 * k + 2], hi[4 * k + 3]);
                        nst += (own_lo ? 0u : 1u) + (own_hi ? 0u : 1u);
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        for (uint32_t j = 0; j < uint32_t(BN / 32); ++j)
                            if (j < own0 || j >= own1)
                                ptx::bulk_store(partial_f4(cluster, 8 * j) - lane, scr + 4096u * j, 4096u);
                        ptx::bulk_commit_group();
                        ptx::bulk_wait_group_all();          // the partials are in global memory
                        ptx::fence_proxy_async_global();
                        __threadfence();
                        ptx::st_release_u64(p.flags + (size_t(cluster) * NCTA + rank) * kEpiWarps + q, p.launch_id);
                    }
                    // 2-3. wait for the other pieces, then load their partials of this slice
                    uint32_t okf = 1;
                    if (lane == 0) {
                        for (uint32_t i = 0; i < np && okf; ++i)
                            if (i != pc)
                                okf = wait_flag(p.flags + (size_t(first + i) * NCTA + rank) * kEpiWarps + q,
                                                p.launch_id, wi, kSiteStreamK) ? 1u : 0u;
                        if (okf) {
                            ptx::fence_proxy_async_global();
                            const uint32_t nown = own1 - own0;
                            const uint32_t xb = ptx::smem_u32(&ctl->xfer[q]);
                            ptx::mbar_arrive_expect_tx(xb, (np - 1) * nown * 4096u);
                            for (uint32_t i = 0, slot = 0; i < np; ++i) {
                                if (i == pc) continue;
                                for (uint32_t jj = 0; jj < nown; ++jj)
                                    ptx::bulk_load(scr + (slot * nown + jj) * 4096u,
                                                   partial_f4(first + i, 8 * (own0 + jj)) - lane, 4096u, xb);
                                ++slot;
                            }
                        }
                    }
                    okf = __shfl_sync(0xffffffffu, okf, 0);
                    (void)nst;
                    if (!okf) break;
                    // every lane observes the loads' completion (each reads the scratch)
                    if (!wait(ptx::smem_u32(&ctl->xfer[q]), 0, wi, kSiteStreamK)) break;
                    const int32_t r = row0 + int32_t(lane);
                    const uint32_t nown = own1 - own0;
#pragma unroll 1
                    for (uint32_t jj = 0; jj < nown; ++jj) {
                        const uint32_t j = own0 + jj;
                        uint32_t v[32];
                        ptx::tmem_ld_32x32b_x32(tacc + 32 * j, v);
                        ptx::tmem_wait_ld();
                        ptx::reg_fence(v);
                        float sum[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) sum[e] = 0.0f;
                        for (uint32_t i = 0, slot = 0; i < np; ++i) {
                            if (i == pc) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) sum[e] += __uint_as_float(v[e]);
                                continue;
                            }
                            const uint32_t blk = scr + (slot * nown + jj) * 4096u;
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                float4 t;
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(t.x), "=f"(t.y), "=f"(t.z), "=f"(t.w)
                                             : "r"(blk + (uint32_t(k) * 32u + lane) * 16u) : "memory");
                                sum[4 * k] += t.x;
                                sum[4 * k + 1] += t.y;
                                sum[4 * k + 2] += t.z;
                                sum[4 * k + 3] += t.w;
                            }
                            ++slot;
                        }
                        uint32_t h[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            h[e] = Cfg::kBF ? ptx::pack_bf16x2_rn(__float_as_uint(sum[2 * e]), __float_as_uint(sum[2 * e + 1]))
                                            : ptx::pack_f16x2_rn(__float_as_uint(sum[2 * e]), __float_as_uint(sum[2 * e + 1]));
                        // 32 columns of this lane's row, in 16-byte pieces where all 8 fit in N
                        if (r < p.M) {
                            uint16_t* crow = p.C + int64_t(r) * p.ldc;
#pragma unroll
                            for (int g8 = 0; g8 < 4; ++g8) {
                                const int32_t n = col0 + int32_t(j) * 32 + g8 * 8;
                                if (n + 8 <= p.N) {
                                    *reinterpret_cast<uint4*>(crow + n) =
                                        make_uint4(h[4 * g8], h[4 * g8 + 1], h[4 * g8 + 2], h[4 * g8 + 3]);
                                } else {
                                    for (int e = 0; e < 8 && n + e < p.N; ++e)
                                        crow[n + e] = uint16_t(h[4 * g8 + e / 2] >> (16 * (e & 1)));
                                }
                            }
                        }
                    }
                    // The last read of this accumulator is done: hand it back.
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (CG == 2) ptx::mbar_arrive_cluster(acce_tgt + 8 * acc);
                        else ptx::mbar_arrive(acce0 + 8 * acc);
                    }
                    if (tr) {
                        tr[5] = ptx::globaltimer();
                        tr[6] = tr[5];
                    }
                    acc ^= 1u;
                    if (acc == 0) acc_phase ^= 1u;
                    continue;
                }
            }
            // An owner adds the partials of the clusters that took the rest of its tile.
            uint32_t npart = 0;
            if (it.kind == kItemOwner) {
                npart = owner_partners(p, it.tile, cluster, nclusters);
                uint32_t okf = 1;
                if (lane == 0)
                    for (uint32_t i = 0; i < npart && okf; ++i)
                        okf = wait_flag(p.flags + (size_t(cluster + 1 + i) * NCTA + rank) * kEpiWarps + q,
                                        p.launch_id, wi, kSiteStreamK) ? 1u : 0u;
                okf = __shfl_sync(0xffffffffu, okf, 0);
                if (!okf) break;
                __threadfence();
            }
            if (tr) tr[5] = ptx::globaltimer();
            const uint32_t tacc = tmem_base + lane_off + acc * uint32_t(BN);
#pragma unroll 1
            for (int c = 0; c < nchunks; ++c) {
                uint32_t lo[32], hi[32];
                ptx::tmem_ld_32x32b_x32(tacc + uint32_t(c * kEpiCols), lo);
                ptx::tmem_ld_32x32b_x32(tacc + uint32_t(c * kEpiCols + 32), hi);
                ptx::tmem_wait_ld();
                ptx::reg_fence(lo);
                ptx::reg_fence(hi);
                if (c == nchunks - 1) {
                    // The whole accumulator is in registers: hand the buffer back.
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (CG == 2) ptx::mbar_arrive_cluster(acce_tgt + 8 * acc);
                        else ptx::mbar_arrive(acce0 + 8 * acc);
                    }
                }
                if (it.kind == kItemPartialOut) {
                    // fp32 partial: 16 float4 groups of this lane's row, 64 columns
                    float4* dst = partial_f4(cluster, uint32_t(c * kEpiCols / 4));
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        __stcg(dst + size_t(j) * 32u,
                               make_float4(__uint_as_float(lo[4 * j]), __uint_as_float(lo[4 * j + 1]),
                                           __uint_as_float(lo[4 * j + 2]), __uint_as_float(lo[4 * j + 3])));
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        __stcg(dst + size_t(8 + j) * 32u,
                               make_float4(__uint_as_float(hi[4 * j]), __uint_as_float(hi[4 * j + 1]),
                                           __uint_as_float(hi[4 * j + 2]), __uint_as_float(hi[4 * j + 3])));
                    continue;
                }
                for (uint32_t i = 0; i < npart; ++i) {   // k order: this piece, then each partner
                    const float4* src = partial_f4(cluster + 1 + i, uint32_t(c * kEpiCols / 4));
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 v = __ldcg(src + size_t(j) * 32u);
                        lo[4 * j] = __float_as_uint(__uint_as_float(lo[4 * j]) + v.x);
                        lo[4 * j + 1] = __float_as_uint(__uint_as_float(lo[4 * j + 1]) + v.y);
                        lo[4 * j + 2] = __float_as_uint(__uint_as_float(lo[4 * j + 2]) + v.z);
                        lo[4 * j + 3] = __float_as_uint(__uint_as_float(lo[4 * j + 3]) + v.w);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 v = __ldcg(src + size_t(8 + j) * 32u);
                        hi[4 * j] = __float_as_uint(__uint_as_float(hi[4 * j]) + v.x);
                        hi[4 * j + 1] = __float_as_uint(__uint_as_float(hi[4 * j + 1]) + v.y);
                        hi[4 * j + 2] = __float_as_uint(__uint_as_float(hi[4 * j + 2]) + v.z);
                        hi[4 * j + 3] = __float_as_uint(__uint_as_float(hi[4 * j + 3]) + v.w);
                    }
                }
                uint32_t h[32];
                if constexpr (Cfg::kA16) {
                    // fp16 accumulator: each column's low half already is the result
#pragma unroll
                    for (int j = 0; j < 16; ++j) h[j] = (lo[2 * j] & 0xFFFFu) | (lo[2 * j + 1] << 16);
#pragma unroll
                    for (int j = 0; j < 16; ++j) h[16 + j] = (hi[2 * j] & 0xFFFFu) | (hi[2 * j + 1] << 16);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        h[j] = Cfg::kBF ? ptx::pack_bf16x2_rn(lo[2 * j], lo[2 * j + 1])
                                        : ptx::pack_f16x2_rn(lo[2 * j], lo[2 * j + 1]);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        h[16 + j] = Cfg::kBF ? ptx::pack_bf16x2_rn(hi[2 * j], hi[2 * j + 1])
                                             : ptx::pack_f16x2_rn(hi[2 * j], hi[2 * j + 1]);
                }

                // The staging buffer about to be written was last read by the
                // store issued two chunks ago.
                if (lane == 0) ptx::bulk_wait_group_read<1>();
                __syncwarp();
                const uint32_t buf = out0 + ob * kOutBufBytes;
                const uint32_t row = buf + lane * 128u;
#pragma unroll
                for (uint32_t j = 0; j < 8; ++j)   // 16-byte chunk j of this row, 128-byte swizzle
                    ptx::st_shared_v4(row + ((j ^ (lane & 7u)) << 4), h[4 * j], h[4 * j + 1],
                                      h[4 * j + 2], h[4 * j + 3]);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                const int32_t cx = col0 + c * kEpiCols;
                if (lane == 0) {
                    // The tensor map spans only the 16-byte-aligned columns [0, N8).
                    if (row0 < p.M && cx < p.N8) ptx::tma_store_2d(&p.tmC, cx, row0, buf);
                    ptx::bulk_commit_group();
                }
                if (p.N8 < p.N && cx <= p.N8 && p.N8 < cx + kEpiCols) {
                    // The last N - N8 (< 8) columns: this lane's row, straight from registers.
                    const int32_t r = row0 + int32_t(lane);
                    if (r < p.M) {
                        uint16_t* dst = p.C + int64_t(r) * p.ldc;
                        for (int32_t e = p.N8; e < p.N; ++e) {
                            // element idx of this lane's staged row (16-byte chunk idx/8, swizzled)
                            const uint32_t idx = uint32_t(e - cx);
                            dst[e] = ptx::ld_shared_u16(row + ((((idx >> 3) ^ (lane & 7u)) << 4) |
                                                               ((idx & 7u) << 1)));
                        }
                    }
                }
                ob ^= 1u;
            }
            if (it.kind == kItemPartialOut) {
                // publish: every lane's partial stores before the flag
                __threadfence();
                __syncwarp();
                if (lane == 0)
                    ptx::st_release_u64(p.flags + (size_t(cluster) * NCTA + rank) * kEpiWarps + q, p.launch_id);
            }
            if (tr) tr[6] = ptx::globaltimer();
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (lane == 0) ptx::bulk_wait_group_all();
        __syncwarp();
    }

    ptx::tc_fence_before();
    if constexpr (NCTA > 1) ptx::cluster_sync(); else __syncthreads();
    ptx::tc_fence_after();
    if (warp == 1) ptx::tmem_dealloc<CG>(tmem_base, Cfg::kTmemCols);
}

// K == 0: the empty sum, +0 over the M×N window.
__global__ void zero_fill_kernel(uint16_t* C, int64_t M, int64_t N, int64_t ldc) {
    const int64_t total = M * N;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t m = i / N, n = i - m * N;
        C[m * ldc + n] = 0;
    }
}

}  // namespace g16
