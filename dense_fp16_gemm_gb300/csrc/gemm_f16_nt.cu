// GB300 (sm_103a) dense fp16 NT GEMM library, C[M,N] = A[M,K] · B[N,K]ᵀ: the
// host side and the C ABI (include/gemm_f16_nt.h).
//
// Two kernels do the work: the persistent, warp-specialised tcgen05 kernel
// (persistent.cuh) and the small-problem kernel (small_tile.cuh).  This file
// checks the arguments, plans each call (which kernel, tile shape, CTA group,
// work schedule: whole tiles, a stream-K split of the last wave, split
// pieces, column slices), encodes the TMA tensor maps, reserves the split's
// workspace once per device, launches with programmatic dependent launch and
// cluster dimensions, and reads back the device watchdog word.  Nothing is
// allocated per call.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "gemm_f16_nt.h"
#include "ptx.cuh"
#include "sched.cuh"

#define G16_EXPORT extern "C" __attribute__((visibility("default")))

#include "persistent.cuh"
#include "small_tile.cuh"

namespace g16 {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

using Cfg2 = KCfg<2, 256, 6>;      // CTA pair, 256×256 tile, 6-stage ring
using Cfg1 = KCfg<1, 256, 4>;      // single CTA, 128×256 tile, 4-stage ring
using Cfg2Bf = KCfg<2, 256, 6, 1, true>;    // the same with bf16 operands and result
using Cfg1Bf = KCfg<1, 256, 4, 1, true>;
using Cfg2A16 = KCfg<2, 256, 6, 1, false, true>;   // the fp16 ones with an fp16 accumulator
using Cfg1A16 = KCfg<1, 256, 4, 1, false, true>;
// The small-problem kernel's tiles: 128·CG × BN, one per cluster (each also
// built for bf16 and for split-K: SCfg's last two parameters), with as many
// ring stages as fit in a CTA's shared memory: the main loop streams the
// operands at what one SM ingests with the ring's bytes in flight (measured,
// µs added after an L2 flush: 1024³ 4.8 with 9 stages against 5.2 with 8,
// 512×4096×4096 16.7 with 7 against 18.4 with 6).
using S1n32 = SCfg<1, 32, 11>;
using S1n64 = SCfg<1, 64, 9>;
using S1n128 = SCfg<1, 128, 7>;
using S2n32 = SCfg<2, 32, 12>;
using S2n64 = SCfg<2, 64, 11>;
using S2n128 = SCfg<2, 128, 9>;
#if G16_MCAST_LIB
using Cfg2x2 = KCfg<2, 256, 6, 2>; // two CTA pairs per cluster sharing A: 256×512 cluster tile
using Cfg2x2Bf = KCfg<2, 256, 6, 2, true>;
using Cfg2x2A16 = KCfg<2, 256, 6, 2, false, true>;
#endif

template <class Cfg>
bool allow_smem() {
    return cudaFuncSetAttribute(gemm_f16_nt_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg::kSmemBytes) == cudaSuccess;
}
template <class... Cfgs>
bool allow_smem_small() {
    return ((cudaFuncSetAttribute(gemm_f16_nt_small_kernel<Cfgs>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  Cfgs::kSmemBytes) == cudaSuccess) && ...);
}
// every small-kernel configuration of one operand type, with and without split-K
template <bool BF, bool SP>
bool allow_smem_small_all() {
    return allow_smem_small<SCfg<1, 32, S1n32::kStages, BF, SP>, SCfg<1, 64, S1n64::kStages, BF, SP>,
                            SCfg<1, 128, S1n128::kStages, BF, SP>, SCfg<2, 32, S2n32::kStages, BF, SP>,
                            SCfg<2, 64, S2n64::kStages, BF, SP>, SCfg<2, 128, S2n128::kStages, BF, SP>>();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A stream-K workspace reserved at a device's set-up.  A launch that uses it
// makes its stream wait for the slot's previous user (`done`), so launches on
// unordered streams that land on the same slot run one after the other; the
// mutex keeps host threads from interleaving wait, launch and record.
struct WorkspaceSlot {
    void* ptr = nullptr;
    cudaEvent_t done = nullptr;
    std::mutex mu;
};
constexpr int kMaxWorkspaceSlots = 8;
constexpr int kDefaultWorkspaceSlots = 4;

struct DeviceState {
    bool ready = false;
    gemm_status_t status = GEMM_OK;
    int sms = 0;
    int max_clusters2 = 0;   // resident CTA pairs for Cfg2
    int max_clusters4 = 0;   // resident clusters of two pairs for Cfg2x2 (0 without it)
    int max_ctas1 = 0;       // resident CTAs for Cfg1
    bool single_gpu = false; // the process sees exactly one CUDA device
    uint32_t* watchdog = nullptr;
    unsigned long long* claim_words = nullptr;   // g_claim_words on this device
    bool ws_ready = false;
    int ws_slots = 0;        // workspace slots reserved (0: stream-K unavailable)
    int64_t ws_bytes = 0;    // bytes per slot
    WorkspaceSlot slot[kMaxWorkspaceSlots];
    std::atomic<uint32_t> next_slot{0};
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
std::atomic<uint64_t> g_launch_seq{0};

constexpr int kMinSplitKb = 8;   // smallest stream-K share worth its fix-up, in k-blocks
constexpr int kTailSplitGainKb = 32;    // k-blocks a split of the last wave must save each cluster
constexpr int kMaxSplitPieces = 8;      // split pieces per tile with fewer tiles than clusters ...
constexpr int kMinPieceKb = 2;          // ... each at least this many k-blocks long,
constexpr int kSplitPiecesMinKb = 48;   // ... taken by default from this k depth (k-blocks)
constexpr int kTailSplitIdlePct = 8;    // idle tile slots (%) above which the last wave may be split
constexpr int kSplitTailMaxKb = 32;     // deepest k for which the default N-splits a last wave
constexpr int64_t kAltKStripBytes = 60000000;   // a round's A and B strips above which k order alternates

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

gemm_status_t setup_device(int dev, DeviceState& st) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (!allow_smem<Cfg2>() || !allow_smem<Cfg1>() || !allow_smem<Cfg2Bf>() || !allow_smem<Cfg1Bf>() ||
        !allow_smem<Cfg2A16>() || !allow_smem<Cfg1A16>() ||
        !allow_smem_small_all<false, false>() || !allow_smem_small_all<false, true>() ||
        !allow_smem_small_all<true, false>() || !allow_smem_small_all<true, true>()) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
#if G16_MCAST_LIB
    if (!allow_smem<Cfg2x2>() || !allow_smem<Cfg2x2Bf>() || !allow_smem<Cfg2x2A16>()) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
#endif
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    st.single_gpu = ndev == 1;
    // How many clusters can be resident at once (cluster placement within the
    // GPCs may leave some SMs out: on a 152-SM GB300, 76 pairs but only 36
    // clusters of four).
    auto resident_clusters = [&](auto kernel, int ctas, int smem) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = ctas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(ctas * (sms / ctas), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            n = sms / ctas;
        }
        return n < sms / ctas ? n : sms / ctas;
    };
    st.max_clusters2 = resident_clusters(gemm_f16_nt_kernel<Cfg2>, 2, Cfg2::kSmemBytes);
#if G16_MCAST_LIB
    st.max_clusters4 = resident_clusters(gemm_f16_nt_kernel<Cfg2x2>, 4, Cfg2x2::kSmemBytes);
#else
    st.max_clusters4 = 0;
#endif
    {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_f16_nt_kernel<Cfg1>, kThreads,
                                                          Cfg1::kSmemBytes) != cudaSuccess ||
            per_sm < 1) {
            cudaGetLastError();
            per_sm = 1;
        }
        st.max_ctas1 = sms;   // one CTA per SM: each holds all 512 TMEM columns
    }
    void* wd = nullptr;
    if (cudaGetSymbolAddress(&wd, g_watchdog_word) != cudaSuccess || !wd) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    st.watchdog = static_cast<uint32_t*>(wd);
    void* cw = nullptr;
    if (cudaGetSymbolAddress(&cw, g_claim_words) != cudaSuccess || !cw) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    st.claim_words = static_cast<unsigned long long*>(cw);
    st.sms = sms;
    return GEMM_OK;
}

// Stream-K workspace: flags first ([cluster][rank][warp] uint64, 256-byte
// aligned), then the fp32 partial tiles ([cluster][rank][256/4][128] float4),
// one 128×256 partial per CTA of the cluster.
constexpr int kCtaTileN = 256;
int64_t flags_bytes(int ctas, int64_t clusters) {
    return (clusters * ctas * kEpiWarps * 8 + 255) / 256 * 256;
}
int64_t workspace_bytes(int ctas, int64_t clusters) {
    return flags_bytes(ctas, clusters) + clusters * ctas * int64_t(kBlockM) * kCtaTileN * 4;
}
// The small-problem kernel's split-K workspace: the same flags, then one
// 128 × bn fp32 partial tile per CTA.
int64_t small_workspace_bytes(int ctas, int bn, int64_t clusters) {
    return flags_bytes(ctas, clusters) + clusters * ctas * int64_t(kBlockM) * bn * 4;
}

// Workspace slots to reserve: GEMM_F16_NT_WORKSPACE_SLOTS (0..8) if set to a
// number, else 4.
int workspace_slots_setting() {
    const char* e = getenv("GEMM_F16_NT_WORKSPACE_SLOTS");
    if (!e || !*e) return kDefaultWorkspaceSlots;
    char* end = nullptr;
    const long v = strtol(e, &end, 10);
    if (end == e || *end != '\0' || v < 0) return kDefaultWorkspaceSlots;
    return v > kMaxWorkspaceSlots ? kMaxWorkspaceSlots : int(v);
}

// Reserve the stream-K workspace slots, each large enough for any launch on
// this device.  If the memory cannot be had, no slot is kept and every call
// is planned without the split (reported in the plan's split_k_off).
void setup_workspace(DeviceState& st) {
    int64_t need = workspace_bytes(2, st.max_clusters2);
    if (workspace_bytes(1, st.max_ctas1) > need) need = workspace_bytes(1, st.max_ctas1);
    if (workspace_bytes(4, st.max_clusters4) > need) need = workspace_bytes(4, st.max_clusters4);
    for (int cg = 1; cg <= 2; ++cg)   // the small kernel's split-K: at most one wave of 128-wide tiles
        if (small_workspace_bytes(cg, 128, st.sms / cg) > need) need = small_workspace_bytes(cg, 128, st.sms / cg);
    const int want = workspace_slots_setting();
    int got = 0;
    for (; got < want; ++got) {
        WorkspaceSlot& sl = st.slot[got];
        if (cudaMalloc(&sl.ptr, size_t(need)) != cudaSuccess) {
            cudaGetLastError();
            sl.ptr = nullptr;
            break;
        }
        if (cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(sl.ptr);
            sl.ptr = nullptr;
            sl.done = nullptr;
            break;
        }
    }
    if (got < want) {   // all or nothing: a partial reservation hides a memory shortage
        for (int i = 0; i < got; ++i) {
            cudaEventDestroy(st.slot[i].done);
            cudaFree(st.slot[i].ptr);
            st.slot[i].ptr = nullptr;
            st.slot[i].done = nullptr;
        }
        got = 0;
    }
    st.ws_slots = got;
    st.ws_bytes = got ? need : 0;
}

// The current device's state after its one-time set-up; `with_workspace` also
// reserves the stream-K workspace slots (the static-scratch entry point never
// needs them).
gemm_status_t device_state(DeviceState** out, int* dev_out, bool with_workspace) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GEMM_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        st.status = setup_device(dev, st);
        st.ready = true;
    }
    if (st.status != GEMM_OK) return st.status;
    if (with_workspace && !st.ws_ready) {
        setup_workspace(st);
        st.ws_ready = true;
    }
    *out = &st;
    if (dev_out) *dev_out = dev;
    return GEMM_OK;
}

gemm_status_t current_device(DeviceState** out, int* dev = nullptr) { return device_state(out, dev, true); }

gemm_status_t check_args(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                         const uint16_t* B, int64_t ldb, const uint16_t* C, int64_t ldc,
                         bool a_mn = false, bool b_mn = false) {
    const int64_t lim = int64_t(1) << 31;
    if (M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMM_OK;
    const int64_t ld_lim = int64_t(1) << 39;   // TMA strides stay below 2^40 bytes
    if (!C || ldc < N || ldc >= ld_lim) return GEMM_ERR_INVALID_VALUE;
    if (K > 0) {
        // a row of A holds K elements ([M, K]) or M ([K, M]); likewise B
        if (!A || !B || lda < (a_mn ? M : K) || ldb < (b_mn ? N : K) || lda >= ld_lim || ldb >= ld_lim)
            return GEMM_ERR_INVALID_VALUE;
        if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
            (lda & 7) || (ldb & 7))
            return GEMM_ERR_MISALIGNED;
    }
    if ((reinterpret_cast<uintptr_t>(C) & 15) || (ldc & 7)) return GEMM_ERR_MISALIGNED;
    return GEMM_OK;
}

// Default CTA pairs per cluster.  In the multicast library, two pairs that
// share A pay off when a row pitch of A or B is not a multiple of 128 bytes:
// every 128-byte row slice of a tile then spans two L2 lines, L2 traffic
// becomes the limit, and halving A's share outweighs the SMs that clusters of
// four leave idle.  They need N wide enough for both pairs' tiles.  The
// default library has one pair per cluster only.
int auto_cluster_pairs(int cg, int64_t N, int64_t lda, int64_t ldb) {
    if (!G16_MCAST_LIB || cg != 2 || N <= kCtaTileN) return 1;
    return (lda % 64 != 0 || ldb % 64 != 0) ? 2 : 1;
}

#if G16_MCAST_LIB
// The multicast library's rule: its tensor maps may cover only this GPU's own
// memory, in a process that sees one GPU.  A and B (first and last element)
// must be device memory of the current device.
gemm_status_t check_local_operands(const DeviceState& st, int dev, int64_t M, int64_t N, int64_t K,
                                   const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                                   bool a_mn, bool b_mn) {
    if (!st.single_gpu) return GEMM_ERR_NOT_LOCAL;
    if (K == 0 || M == 0 || N == 0) return GEMM_OK;   // no operand is read
    const int64_t a_rows = a_mn ? K : M, a_cols = a_mn ? M : K;
    const int64_t b_rows = b_mn ? K : N, b_cols = b_mn ? N : K;
    const void* ends[4] = {A, A + (a_rows - 1) * lda + (a_cols - 1), B, B + (b_rows - 1) * ldb + (b_cols - 1)};
    for (const void* q : ends) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_NOT_LOCAL;
        }
        if (at.type != cudaMemoryTypeDevice || at.device != dev) return GEMM_ERR_NOT_LOCAL;
    }
    return GEMM_OK;
}
#endif

// The options with every "auto" (zero) CTA-group and cluster choice resolved.
gemm_f16_nt_options_t resolve_options(const gemm_f16_nt_options_t* o, int64_t N, int64_t lda, int64_t ldb) {
    gemm_f16_nt_options_t r = o ? *o : gemm_f16_nt_options_t{};
    // cta_group stays 0 (automatic): the plan picks the small-problem kernel's
    // CTA group itself; the persistent kernel reads 0 as 2.
    if (r.cluster_pairs == 0) r.cluster_pairs = auto_cluster_pairs(r.cta_group ? r.cta_group : 2, N, lda, ldb);
    return r;
}

int resident_clusters_for(const DeviceState& st, const gemm_f16_nt_options_t& r) {
    return r.cta_group == 1 ? st.max_ctas1 : (r.cluster_pairs == 2 ? st.max_clusters4 : st.max_clusters2);
}

// ---- the small-problem kernel's plan ----

bool small_tile_n_valid(int tn) { return tn == 0 || tn == 32 || tn == 64 || tn == 128; }

// Ring depth, shared memory, tensor-memory columns and most split-K pieces of
// SCfg<cg, bn>.
void small_cfg_info(int cg, int bn, int32_t* stages, int32_t* smem, int32_t* tmem, int32_t* max_pieces) {
#define G16_SMALL_INFO(C, N, T)                  \
    if (cg == C && bn == N) {                     \
        *stages = T::kStages;                     \
        *smem = T::kSmemBytes;                    \
        *tmem = T::kTmemCols;                     \
        *max_pieces = T::kMaxPieces;              \
        return;                                   \
    }
    G16_SMALL_INFO(1, 32, S1n32)
    G16_SMALL_INFO(1, 64, S1n64)
    G16_SMALL_INFO(1, 128, S1n128)
    G16_SMALL_INFO(2, 32, S2n32)
    G16_SMALL_INFO(2, 64, S2n64)
    G16_SMALL_INFO(2, 128, S2n128)
#undef G16_SMALL_INFO
    *stages = *smem = *tmem = *max_pieces = 0;
}

// The small kernel's automatic tile width: the narrowest of 32, 64 and 128
// columns whose 128·cg × bn tiles fit on the SMs in one wave (more, smaller
// tiles: less of A and B for each SM to load, less k-loop per tile), 0 if none
// does.  Measured on GB300 (L2 flushed, time the GEMM adds after a flush): at
// 256³ 32-wide tiles on 16 SMs took 2.2 us against 3.0 (64) and 4.1 (128); at
// 1024³, where 32-wide tiles need two waves, 64-wide ones 6.1 us against 10.3.
int small_tile_n(int64_t M, int64_t N, int cg, int32_t num_sms) {
    const int64_t slots = num_sms / cg;
    const int64_t mt = cdiv(M, int64_t(kBlockM) * cg);
    for (int bn = 32; bn <= 128; bn *= 2)
        if (mt * cdiv(N, bn) <= slots) return bn;
    return 0;
}

// Deepest k per CTA (in 64-wide k-blocks) for which the automatic plan takes the
// small kernel; deeper problems go to the persistent kernel.
constexpr int64_t kSmallMaxKb = 128;
// Split-K in the small kernel: each piece at least kSmallMinPieceKb k-blocks
// long, all tiles' pieces in one wave, at most as many pieces as the owner can
// take the others' partials of into its idle ring at once (8 for 32-wide
// tiles, 4 for 64- and 128-wide ones).
constexpr int64_t kSmallMinPieceKb = 8;
// ... and only from kSmallMinSplitKb k-blocks: the exchange of partials costs
// about 2.5 us (write, flag, load back: L2 round trips), about 15 k-blocks of
// a piece's main loop.  Measured at 256×256×1024 (16 k-blocks): 9.5 us in two
// pieces.
constexpr int64_t kSmallMinSplitKb = 32;

// The number of split-K pieces per tile: the largest power of two within
// those limits.  Few tiles and deep k: at 256×256×4096, 16 tiles of 128×32
// and 64 k-blocks become 128 pieces of 8.
int64_t small_pieces(int64_t tiles, int64_t kb, int cg, int bn, int32_t num_sms) {
    int32_t st, sm, tm, max_pieces;
    small_cfg_info(cg, bn, &st, &sm, &tm, &max_pieces);
    const int64_t slots = num_sms / cg;
    int64_t s = 1;
    while (kb >= kSmallMinSplitKb && s < max_pieces && tiles * s * 2 <= slots && kb >= s * 2 * kSmallMinPieceKb)
        s *= 2;
    return s;
}

// Whether the automatic plan takes the small-problem kernel: every automatic
// option (no CTA group, schedule, raster, grid or tile width asked for), the
// kernel's operand forms, one wave of tiles and k no deeper than kSmallMaxKb.
// Where it applies, the persistent kernel would leave most CTA pairs idle.
// Measured against the persistent kernel's default plan (us, L2 flushed):
// 256³ 2.2 against 6.1, 1024³ 6.1 against 10.2, 512×4096×4096 18.7 against
// 26.5, 128×4096×4096 14.4 against 22.7, 1024×1024×8192 26.7 against 26.9;
// 2048³ and 4096×1024×1024 need more than one wave and stay persistent.
bool small_kernel_pays(int64_t M, int64_t N, int64_t K, const gemm_f16_nt_options_t* o, bool small_ok,
                       int32_t num_sms) {
    if (!small_ok) return false;
    if (o && (o->cta_group != 0 || o->swizzle != 0 || o->max_clusters != 0 || o->schedule != 0 ||
              o->cluster_pairs > 1 || o->tile_n != 0))
        return false;
    const int bn = small_tile_n(M, N, 1, num_sms);
    if (bn == 0) return false;
    const int64_t tiles = cdiv(M, kBlockM) * cdiv(N, bn), kb = cdiv(K, kBlockK);
    return cdiv(kb, small_pieces(tiles, kb, 1, bn, num_sms)) <= kSmallMaxKb;
}

gemm_status_t small_plan(int64_t M, int64_t N, int64_t K, int cg, int bn, int32_t num_sms, bool allow_split_k,
                         gemm_f16_nt_plan_t* pl) {
    memset(pl, 0, sizeof(*pl));
    const int64_t mt = cdiv(M, int64_t(kBlockM) * cg), nt = cdiv(N, bn);
    const int64_t tiles = mt * nt;
    if (tiles * cg >= (int64_t(1) << 31)) return GEMM_ERR_INVALID_VALUE;
    const int64_t kb = cdiv(K, kBlockK);
    const int64_t pieces = allow_split_k ? small_pieces(tiles, kb, cg, bn, num_sms) : 1;
    pl->kernel = 1;
    pl->cta_group = cg;
    pl->cluster_pairs = 1;
    pl->tile_m = kBlockM * cg;
    pl->tile_n = bn;
    pl->block_k = kBlockK;
    int32_t max_pieces = 0;
    small_cfg_info(cg, bn, &pl->stages, &pl->smem_bytes, &pl->tmem_cols, &max_pieces);
    pl->m_tiles = int32_t(mt);
    pl->n_tiles = int32_t(nt);
    pl->k_blocks = int32_t(cdiv(K, kBlockK));
    pl->num_tiles = tiles;
    pl->swizzle = 1;
    pl->clusters = int32_t(tiles * pieces);
    pl->grid_ctas = int32_t(tiles * pieces * cg);
    pl->tail_split = 1;
    pl->split_pieces = int32_t(pieces);
    pl->workspace_bytes = pieces > 1 ? small_workspace_bytes(cg, bn, tiles * pieces) : 0;
    return GEMM_OK;
}

gemm_status_t make_plan(int64_t M, int64_t N, int64_t K, int32_t num_sms, int32_t max_resident,
                        const gemm_f16_nt_options_t* o, gemm_f16_nt_plan_t* pl,
                        bool allow_split_k = true) {
    const int64_t lim = int64_t(1) << 31;
    if (!pl || M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim || num_sms < 1)
        return GEMM_ERR_INVALID_VALUE;
    const int cg = (o && o->cta_group) ? o->cta_group : 2;
    const int sw = (o && o->swizzle) ? o->swizzle : kDefaultSwizzle;
    const int sched = o ? o->schedule : 0;
    const int cp = (o && o->cluster_pairs) ? o->cluster_pairs : 1;
    const int acc = o ? o->accumulate : 0;
    const int tn = o ? o->tile_n : 0;
    if ((cg != 1 && cg != 2) || sw < 1 || sw > 64 || (o && o->max_clusters < 0) || sched < 0 ||
        sched > 5 || cp < 1 || cp > 2 || (cp == 2 && (cg != 2 || !G16_MCAST_LIB)) || acc < 0 || acc > 1 ||
        !small_tile_n_valid(tn))
        return GEMM_ERR_INVALID_VALUE;
    // The small-problem kernel: K-major A and B, fp32 accumulator, one pair
    // (or CTA) per cluster, no trace.
    const bool small_ok = cp == 1 && acc == 0 && !(o && (o->a_layout != 0 || o->b_layout != 0 || o->trace));
    if (sched == 5 && !small_ok) return GEMM_ERR_INVALID_VALUE;
    if (sched == 5 || (K > 0 && small_kernel_pays(M, N, K, o, small_ok, num_sms))) {
        const int scg = (o && o->cta_group) ? o->cta_group : 1;
        int bn = tn ? tn : small_tile_n(M, N, scg, num_sms);
        if (bn == 0) bn = 128;   // forced on a problem too large for one wave: widest tiles
        return small_plan(M, N, K, scg, bn, num_sms, allow_split_k && acc == 0, pl);
    }
    memset(pl, 0, sizeof(*pl));
    pl->cta_group = cg;
    pl->cluster_pairs = cp;
    pl->tile_m = kBlockM * cg;
    pl->tile_n = kCtaTileN * cp;
    pl->block_k = kBlockK;
    pl->stages = cg == 2 ? Cfg2::kStages : Cfg1::kStages;
    pl->smem_bytes = cg == 2 ? Cfg2::kSmemBytes : Cfg1::kSmemBytes;
    pl->tmem_cols = cg == 2 ? Cfg2::kTmemCols : Cfg1::kTmemCols;
    const int64_t mt = cdiv(M, pl->tile_m), nt = cdiv(N, pl->tile_n);
    const int64_t tiles = mt * nt;
    if (tiles >= lim || mt * sw >= lim) return GEMM_ERR_INVALID_VALUE;
    pl->m_tiles = int32_t(mt);
    pl->n_tiles = int32_t(nt);
    pl->k_blocks = int32_t(cdiv(K, kBlockK));
    pl->num_tiles = tiles;
    pl->swizzle = int32_t(nt > 0 && sw > nt ? nt : sw);
    int64_t resident = max_resident > 0 ? max_resident : num_sms / (cg * cp);
    if (resident < 1) resident = 1;
    if (o && o->max_clusters > 0 && o->max_clusters < resident) resident = o->max_clusters;

    // Schedule.  Whole tiles round-robin over the clusters leave the last wave
    // partly empty when tiles % clusters != 0.  The stream-K part spreads the
    // k-block units of (the partial wave + one full wave) evenly instead; with
    // fewer tiles than clusters it spreads all of them.  Splitting costs fp32
    // partial tiles through L2 (and DRAM), so auto mode (0) splits only when at
    // least kTailSplitIdlePct % of the whole-tile schedule's tile slots would sit
    // idle, with one pair per cluster (two-pair clusters are picked when L2
    // traffic already limits), and every share keeps at least kMinSplitKb
    // k-blocks.  Measured on GB300: 4096^3 (16 % idle) gains 5.6 %,
    // 4096x11008x4096 (9.5 %) 3 %; 6144^3 (5.3 %) ties; 8192^3 (3.8 % idle,
    // power-capped) loses 1.4 % when split.  1 = whole tiles only; 2 = stream-K
    // whenever it can; 3 = N-split whenever it can; 4 = split pieces whenever
    // they can run.
    const int64_t kb = pl->k_blocks;
    int64_t clusters = tiles < resident ? tiles : resident;
    int64_t sk_tiles = 0, tail_tiles = 0, tail_split = 1, split_pieces = 1;
    // An fp16 accumulator never splits in k: that would add fp32 partials of
    // fp16 accumulators, a different rounding sequence.
    if (allow_split_k && tiles > 0 && kb > 0 && sched != 1 && sched != 3 && acc == 0) {
        if (tiles >= resident) {
            // Split only if it spares each cluster >= kSmallSplitGainKb k-blocks
            // (kb·(rounds - tiles/clusters) of them) and at least one full wave
            // of whole tiles remains.  Measured with L2 flushed: 4096^3 (64
            // k-blocks, 256 tiles) 84.9 us split against 90.2 whole; but
            // 4096x4096x1024 (16 k-blocks) 36.7 against 33.5, 3584x2304x2048
            // (32) 36.2 against 31.5, and 2048x4096x8192 (128 tiles, all split)
            // 99.9 against 90.6.
            const int64_t rem = tiles % resident;
            const int64_t slots = (tiles + resident - 1) / resident * resident;
            const bool deep = kb * (slots - tiles) >= kTailSplitGainKb * resident;
            const bool worth = rem != 0 && cp == 1 && (slots - tiles) * 100 >= kTailSplitIdlePct * slots &&
                               kb >= kMinSplitKb && deep && tiles >= 2 * resident;
            if (sched == 2 || worth) sk_tiles = rem + resident;
            if (sk_tiles > tiles) sk_tiles = tiles;
        } else if (sched == 2) {
            // Forced stream-K with fewer tiles than clusters (tests): all the
            // tiles' k-blocks spread evenly, owners adding their partners'
            // partials one after another.
            int64_t g = tiles * kb;                    // up to one k-block each
            if (g > resident) g = resident;
            if (g > tiles) {
                clusters = g;
                sk_tiles = tiles;
            }
        } else if (cp == 1) {
            // Fewer tiles than clusters: cut every tile along k into s equal
            // split pieces on s clusters, s = 2, 4 or 8 (the largest with
            // tiles·s <= clusters and at least kMinPieceKb k-blocks a piece).
            // The pieces reduce each other's partials in parallel (each owns
            // s-th of the columns), so the fix-up costs one partial round trip
            // through L2 per piece; with (s-1) partial tiles written per tile
            // it is bound by the L2's aggregate write rate (about 5 TB/s
            // measured).  Measured with L2 flushed, default against N-split:
            // 256x256x8192 23.0 us (8 pieces) against 42.6, 1024x1024x8192 29.1
            // (4) against 44.6, 1024x1024x4096 23.0 against 27.1, 512x4096x4096
            // 27.1 (2) against 28.2; but at k = 1024 and 2048 the N-split wins
            // (1024^3 14.8 against 19.0, 768x768x2048 18.0 against 20.0).  So
            // the default takes it from kSplitPiecesMinKb k-blocks.
            const int64_t min_kb = sched == 4 ? 1 : kMinPieceKb;   // forced: pieces of one k-block allowed
            int64_t sp = 1;
            while (sp < kMaxSplitPieces && tiles * sp * 2 <= resident && kb >= sp * 2 * min_kb) sp *= 2;
            if (sp > 1 && (sched == 4 || kb >= kSplitPiecesMinKb)) {
                split_pieces = sp;
                clusters = tiles * sp;
            }
        }
    }
    // N-split: with no stream-K split, the R tiles of a last wave that fills at
    // most half of the clusters (all tiles, with fewer tiles than clusters) are
    // each cut into s = 2 or 4 column slices (the largest with R·s <= clusters)
    // that run on their own pairs.  A narrower MMA is not proportionally faster
    // (with no loads, N = 128 takes 69 % and N = 64 62 % of the 256-wide time
    // per k-block), and with their loads split slices measured no faster than
    // whole tiles, so this does not shorten a compute-bound wave; what it
    // shortens is each cluster's epilogue.  So the default uses
    // it for small problems, and for the last wave only when k is shallow:
    // 4096x4096x1024 ran 31.2 us against 33.5 whole, while at 8192^3 the split
    // last wave measured 693.8 against 688.8 us.  One pair per cluster and B
    // stored [N, K] only.
    const bool can_split = cg == 2 && cp == 1 && !(o && o->b_layout == 1);
    if (sk_tiles == 0 && split_pieces == 1 && tiles > 0 && kb > 0 && can_split &&
        ((sched == 0 && (tiles < resident || kb <= kSplitTailMaxKb)) || sched == 3)) {
        const int64_t R = tiles % resident;          // all tiles when tiles < resident
        int64_t s = 1;
        while (s < 4 && R > 0 && R * s * 2 <= resident) s *= 2;
        if (s > 1) {
            tail_tiles = R;
            tail_split = s;
            clusters = tiles >= resident ? resident : R * s;
        }
    }
    pl->clusters = int32_t(clusters);
    pl->grid_ctas = int32_t(clusters * cg * cp);
    pl->sk_tiles = int32_t(sk_tiles);
    pl->workspace_bytes = (sk_tiles > 0 || split_pieces > 1) ? workspace_bytes(cg * cp, clusters) : 0;
    pl->tail_tiles = int32_t(tail_tiles);
    pl->tail_split = int32_t(tail_split);
    pl->split_pieces = int32_t(split_pieces);
    // k order of whole tiles (item_k_down in sched.cuh).  A round of whole
    // tiles streams the k-slabs of about rows·tile_m rows of A and w·tile_n
    // rows of B (w = the raster group's width, rows = clusters / w).  When
    // those strips do not fit in the part of L2 that holds them, a round that
    // starts again from k-block 0 finds the first slabs evicted by the last,
    // and re-reads both strips from DRAM; alternating the direction per round
    // starts each round on the slabs just read.  An LRU model of L2 fitted to
    // measured DRAM reads at 8192^3 (raster widths 2-32: 1.79-2.06 GB modelled
    // against 1.92-2.10 measured, with 63 MB of effective capacity) puts the
    // gain from about 60 MB of strips: at 8192^3 (75 MB) reads went from 0.968
    // to 0.793 GB a launch, power-capped launches from 692.9 to 682.2 us and
    // bursts from 607.7 to 599.6 us; on the MLP shape (38 MB) it cost 0.3 %.
    // An fp16 accumulator keeps k order (its rounding depends on it).
    // The last, partial wave of whole tiles is claimed at run time: per-cluster
    // tile times differ systematically by about 4 % on this GPU (the same
    // clusters are the slow ones launch after launch), and the static deal
    // gives the extra tile to clusters 0.. whatever their speed.
    pl->claimed_tiles = 0;
    if (allow_split_k && sk_tiles == 0 && tail_split == 1 && split_pieces == 1 && clusters > 0 &&
        tiles > clusters && tiles % clusters != 0)
        pl->claimed_tiles = int32_t(tiles % clusters);
    pl->k_order = 0;
    if (acc == 0 && tiles - sk_tiles > clusters && clusters > 0) {
        const int64_t w = pl->swizzle;
        const int64_t rows = cdiv(clusters, w);
        const int64_t strips_bytes = (rows * pl->tile_m + w * pl->tile_n) * kb * kBlockK * 2;
        if (strips_bytes > kAltKStripBytes) pl->k_order = 1;
    }
    return GEMM_OK;
}

gemm_status_t encode_2d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* ptr, uint64_t inner,
                        uint64_t outer, uint64_t pitch_elems, uint32_t box_inner, uint32_t box_outer) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch_elems * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(tm, dtype, 2, const_cast<void*>(ptr), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_LAUNCH;
}

template <class Cfg>
gemm_status_t launch(const gemm_f16_nt_plan_t& pl, int64_t M, int64_t N, int64_t K, const uint16_t* A,
                     int64_t lda, const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc,
                     cudaStream_t stream, const gemm_f16_nt_options_t* o, uint32_t* watchdog,
                     void* workspace) {
    Params p;
    memset(&p, 0, sizeof(p));
    gemm_status_t s;
    // A TMA store clips the innermost dimension in 16-byte units, so the map for
    // C covers only the first N8 = N - N % 8 columns; the kernel writes the rest
    // with plain stores and no byte past column N-1 is ever written.
    const int64_t N8 = N & ~int64_t(7);
    const CUtensorMapDataType dt = Cfg::kBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const bool a_mn = o && o->a_layout == 1, b_mn = o && o->b_layout == 1;
    if ((s = a_mn ? encode_2d(&p.tmA, dt, A, uint64_t(M), uint64_t(K), uint64_t(lda), 64, 64)
                  : encode_2d(&p.tmA, dt, A, uint64_t(K), uint64_t(M), uint64_t(lda), kBlockK,
                              kBlockM / Cfg::kCP)) != GEMM_OK ||
        (s = b_mn ? encode_2d(&p.tmB, dt, B, uint64_t(N), uint64_t(K), uint64_t(ldb), 64, 64)
                  : encode_2d(&p.tmB, dt, B, uint64_t(K), uint64_t(N), uint64_t(ldb), kBlockK,
                              Cfg::kBRows)) != GEMM_OK ||
        (N8 > 0 && (s = encode_2d(&p.tmC, dt, C, uint64_t(N8), uint64_t(M), uint64_t(ldc), kEpiCols, 32)) != GEMM_OK))
        return s;
    p.N8 = int32_t(N8);
    p.C = C;
    p.ldc = ldc;
    p.raster = make_raster(uint32_t(pl.m_tiles), uint32_t(pl.n_tiles), uint32_t(pl.swizzle));
    set_schedule(p, pl);
    p.M = int32_t(M);
    p.N = int32_t(N);
    p.timeout_ns = (o && o->timeout_ns) ? o->timeout_ns : kDefaultTimeoutNs;
    p.item_timeout_ns = p.timeout_ns + uint64_t(pl.k_blocks) * kItemWaitNsPerKb;
    p.watchdog = watchdog;
    p.inject_stall = o ? o->inject_stall : 0;
    p.a_mn = a_mn ? 1u : 0u;
    p.b_mn = b_mn ? 1u : 0u;
    if (pl.workspace_bytes > 0) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        p.flags = reinterpret_cast<uint64_t*>(ws);
        p.partials = reinterpret_cast<float*>(ws + flags_bytes(Cfg::kCtas, pl.clusters));
    }
    p.launch_id = ++g_launch_seq;
    if (pl.claimed_tiles > 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || !g_dev[dev].claim_words) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
        p.claim = g_dev[dev].claim_words + (p.launch_id % uint64_t(kClaimWords));
    }
    if (pl.tail_split > 1 &&
        (b_mn || Cfg::kCP != 1 ||
         (s = encode_2d(&p.tmBp, dt, B, uint64_t(K), uint64_t(N), uint64_t(ldb), kBlockK,
                        Cfg::kBRows / pl.tail_split)) != GEMM_OK))
        return b_mn || Cfg::kCP != 1 ? GEMM_ERR_INVALID_VALUE : s;
    if (o && o->trace && o->trace_items > 0) {
        p.trace = o->trace;
        p.trace_items = uint32_t(o->trace_items);
    }

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(uint32_t(pl.grid_ctas), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    // may overlap its set-up with the tail of the previous kernel on the stream
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (Cfg::kCtas > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = Cfg::kCtas;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    if (cudaLaunchKernelEx(&cfg, gemm_f16_nt_kernel<Cfg>, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

template <class Cfg>
gemm_status_t launch_small(const gemm_f16_nt_plan_t& pl, int64_t M, int64_t N, int64_t K, const uint16_t* A,
                           int64_t lda, const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc,
                           cudaStream_t stream, const gemm_f16_nt_options_t* o, uint32_t* watchdog,
                           void* workspace) {
    SmallParams p;
    memset(&p, 0, sizeof(p));
    gemm_status_t s;
    const CUtensorMapDataType dt = Cfg::kBF ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if ((s = encode_2d(&p.tmA, dt, A, uint64_t(K), uint64_t(M), uint64_t(lda), kBlockK, kBlockM)) != GEMM_OK ||
        (s = encode_2d(&p.tmB, dt, B, uint64_t(K), uint64_t(N), uint64_t(ldb), kBlockK, Cfg::kBRows)) != GEMM_OK)
        return s;
    p.C = C;
    p.ldc = ldc;
    p.M = int32_t(M);
    p.N = int32_t(N);
    p.m_tiles = uint32_t(pl.m_tiles);
    p.num_kb = uint32_t(pl.k_blocks);
    p.timeout_ns = (o && o->timeout_ns) ? o->timeout_ns : kDefaultTimeoutNs;
    p.item_timeout_ns = p.timeout_ns + uint64_t(pl.k_blocks) * kItemWaitNsPerKb;
    p.watchdog = watchdog;
    p.inject_stall = o ? o->inject_stall : 0;
    p.pieces = uint32_t(pl.split_pieces > 1 ? pl.split_pieces : 1);
    if (p.pieces > 1) {
        if (!workspace) return GEMM_ERR_INVALID_VALUE;
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        p.flags = reinterpret_cast<uint64_t*>(ws);
        p.partials = reinterpret_cast<float*>(ws + flags_bytes(Cfg::kCG, pl.clusters));
    }
    p.launch_id = ++g_launch_seq;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(uint32_t(pl.grid_ctas), 1, 1);
    cfg.blockDim = dim3(kSmallThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (Cfg::kCG == 2) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    if (cudaLaunchKernelEx(&cfg, gemm_f16_nt_small_kernel<Cfg>, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

template <bool BF>
gemm_status_t launch_small_any(const gemm_f16_nt_plan_t& pl, int64_t M, int64_t N, int64_t K, const uint16_t* A,
                               int64_t lda, const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc,
                               cudaStream_t stream, const gemm_f16_nt_options_t* o, uint32_t* watchdog, void* ws) {
#define G16_SMALL_LAUNCH(CG, N_, S_)                                                                    \
    if (pl.cta_group == CG && pl.tile_n == N_)                                                          \
        return pl.split_pieces > 1                                                                      \
                   ? launch_small<SCfg<CG, N_, S_::kStages, BF, true>>(pl, M, N, K, A, lda, B, ldb, C, ldc, \
                                                                        stream, o, watchdog, ws)         \
                   : launch_small<SCfg<CG, N_, S_::kStages, BF, false>>(pl, M, N, K, A, lda, B, ldb, C, ldc, \
                                                                         stream, o, watchdog, ws);
    G16_SMALL_LAUNCH(1, 32, S1n32)
    G16_SMALL_LAUNCH(1, 64, S1n64)
    G16_SMALL_LAUNCH(1, 128, S1n128)
    G16_SMALL_LAUNCH(2, 32, S2n32)
    G16_SMALL_LAUNCH(2, 64, S2n64)
    G16_SMALL_LAUNCH(2, 128, S2n128)
#undef G16_SMALL_LAUNCH
    return GEMM_ERR_INVALID_VALUE;
}

// Why a call ran without the stream-K split that its shape would take
// (gemm_f16_nt_plan_t.split_k_off).
enum : int32_t { kSplitOn = 0, kSplitOffCapture = 1, kSplitOffNoWorkspace = 2 };

gemm_status_t check_options(const gemm_f16_nt_options_t* o, bool bf16) {
    if (!o) return GEMM_OK;
    if (o->a_layout < 0 || o->a_layout > 1 || o->b_layout < 0 || o->b_layout > 1 || o->accumulate < 0 ||
        o->accumulate > 1 || (bf16 && o->accumulate != 0))
        return GEMM_ERR_INVALID_VALUE;
    if ((o->cta_group != 0 && o->cta_group != 1 && o->cta_group != 2) || o->swizzle < 0 || o->swizzle > 64 ||
        o->max_clusters < 0 || o->schedule < 0 || o->schedule > 5 || !small_tile_n_valid(o->tile_n) ||
        o->cluster_pairs < 0 ||
        o->cluster_pairs > (G16_MCAST_LIB ? 2 : 1) || (o->cluster_pairs == 2 && o->cta_group == 1) ||
        o->trace_items < 0 || (o->trace && (reinterpret_cast<uintptr_t>(o->trace) & 7)))
        return GEMM_ERR_INVALID_VALUE;
    return GEMM_OK;
}

// The plan a call on `stream` gets on this device.  A captured launch is
// replayed with the parameters it was captured with; the stream-K split tags
// its completion flags with a per-launch id, which a replay would repeat (an
// owner could then take a partner's partial from an earlier replay), so a call
// made under stream capture runs without it.  Without reserved workspace the
// split is off too.  `split_k_off` records either reason when the shape would
// have split.
gemm_status_t plan_call(const DeviceState& st, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                        const gemm_f16_nt_options_t& ro, bool have_workspace, gemm_f16_nt_plan_t* pl) {
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    const int32_t off = capture != cudaStreamCaptureStatusNone ? kSplitOffCapture
                        : !have_workspace                      ? kSplitOffNoWorkspace
                                                               : kSplitOn;
    const int resident = resident_clusters_for(st, ro);
    gemm_status_t s = make_plan(M, N, K, st.sms, resident, &ro, pl, off == kSplitOn);
    if (s != GEMM_OK || off == kSplitOn) return s;
    gemm_f16_nt_plan_t would;
    if ((s = make_plan(M, N, K, st.sms, resident, &ro, &would, true)) != GEMM_OK) return s;
    if (would.sk_tiles > 0 || would.split_pieces > 1) pl->split_k_off = off;
    return GEMM_OK;
}

template <class C2, class C2x2, class C1>
gemm_status_t launch_cfg(const gemm_f16_nt_plan_t& pl, int64_t M, int64_t N, int64_t K, const uint16_t* A,
                         int64_t lda, const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc,
                         cudaStream_t stream, const gemm_f16_nt_options_t* o, uint32_t* watchdog, void* ws) {
    if (pl.cta_group == 1) return launch<C1>(pl, M, N, K, A, lda, B, ldb, C, ldc, stream, o, watchdog, ws);
    if constexpr (!std::is_void<C2x2>::value)
        if (pl.cluster_pairs == 2) return launch<C2x2>(pl, M, N, K, A, lda, B, ldb, C, ldc, stream, o, watchdog, ws);
    return launch<C2>(pl, M, N, K, A, lda, B, ldb, C, ldc, stream, o, watchdog, ws);
}

#if G16_MCAST_LIB
using Cfg2x2_ = Cfg2x2;
using Cfg2x2Bf_ = Cfg2x2Bf;
using Cfg2x2A16_ = Cfg2x2A16;
#else
using Cfg2x2_ = void;
using Cfg2x2Bf_ = void;
using Cfg2x2A16_ = void;
#endif

gemm_status_t launch_any(bool bf16, const gemm_f16_nt_plan_t& pl, int64_t M, int64_t N, int64_t K,
                         const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc,
                         cudaStream_t stream, const gemm_f16_nt_options_t* ro, uint32_t* watchdog, void* ws) {
    if (pl.kernel == 1)
        return bf16 ? launch_small_any<true>(pl, M, N, K, A, lda, B, ldb, C, ldc, stream, ro, watchdog, ws)
                    : launch_small_any<false>(pl, M, N, K, A, lda, B, ldb, C, ldc, stream, ro, watchdog, ws);
    if (bf16)
        return launch_cfg<Cfg2Bf, Cfg2x2Bf_, Cfg1Bf>(pl, M, N, K, A, lda, B, ldb, C, ldc, stream, ro, watchdog, ws);
    if (ro->accumulate == 1)
        return launch_cfg<Cfg2A16, Cfg2x2A16_, Cfg1A16>(pl, M, N, K, A, lda, B, ldb, C, ldc, stream, ro, watchdog, ws);
    return launch_cfg<Cfg2, Cfg2x2_, Cfg1>(pl, M, N, K, A, lda, B, ldb, C, ldc, stream, ro, watchdog, ws);
}

gemm_status_t zero_fill(const DeviceState& st, int64_t M, int64_t N, uint16_t* C, int64_t ldc,
                        cudaStream_t stream) {
    const int64_t total = M * N;
    int64_t blocks = cdiv(total, 256);
    if (blocks > int64_t(st.sms) * 8) blocks = int64_t(st.sms) * 8;
    zero_fill_kernel<<<dim3(uint32_t(blocks)), dim3(256), 0, stream>>>(C, M, N, ldc);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
}

gemm_status_t run(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, const uint16_t* B,
                  int64_t ldb, uint16_t* C, int64_t ldc, void* stream_v, const gemm_f16_nt_options_t* o,
                  bool bf16 = false) {
    gemm_status_t s = check_options(o, bf16);
    if (s != GEMM_OK) return s;
    const bool a_mn = o && o->a_layout == 1, b_mn = o && o->b_layout == 1;
    if ((s = check_args(M, N, K, A, lda, B, ldb, C, ldc, a_mn, b_mn)) != GEMM_OK) return s;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceState* st = nullptr;
    int dev = -1;
    if ((s = current_device(&st, &dev)) != GEMM_OK) return s;
#if G16_MCAST_LIB
    if ((s = check_local_operands(*st, dev, M, N, K, A, lda, B, ldb, a_mn, b_mn)) != GEMM_OK) return s;
#endif
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    if (K == 0) return zero_fill(*st, M, N, C, ldc, stream);
    const gemm_f16_nt_options_t ro = resolve_options(o, N, lda, ldb);
    gemm_f16_nt_plan_t pl;
    if ((s = plan_call(*st, M, N, K, stream, ro, st->ws_slots > 0, &pl)) != GEMM_OK) return s;
    if (pl.workspace_bytes == 0)
        return launch_any(bf16, pl, M, N, K, A, lda, B, ldb, C, ldc, stream, &ro, st->watchdog, nullptr);
    if (pl.workspace_bytes > st->ws_bytes) return GEMM_ERR_LAUNCH;   // every slot fits any plan of this device
    // A reserved workspace slot, taken round-robin.  The stream first waits for
    // the slot's previous launch (a no-op if it has finished or ran on this
    // stream), so launches on unordered streams never share a slot at the same time.
    WorkspaceSlot& sl = st->slot[st->next_slot.fetch_add(1) % uint32_t(st->ws_slots)];
    std::lock_guard<std::mutex> lock(sl.mu);
    if (cudaStreamWaitEvent(stream, sl.done, 0) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if ((s = launch_any(bf16, pl, M, N, K, A, lda, B, ldb, C, ldc, stream, &ro, st->watchdog, sl.ptr)) != GEMM_OK)
        return s;
    if (cudaEventRecord(sl.done, stream) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

// The plan gemm_f16_nt(_ex) would launch for these arguments on the current
// device and `stream` (its stream-capture state included).
gemm_status_t launch_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, void* stream_v,
                          const gemm_f16_nt_options_t* o, gemm_f16_nt_plan_t* pl) {
    if (!pl) return GEMM_ERR_INVALID_VALUE;
    gemm_status_t s = check_options(o, false);
    if (s != GEMM_OK) return s;
    const int64_t lim = int64_t(1) << 31;
    if (M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim || lda < 0 || ldb < 0)
        return GEMM_ERR_INVALID_VALUE;
    DeviceState* st = nullptr;
    if ((s = current_device(&st)) != GEMM_OK) return s;
    const gemm_f16_nt_options_t ro = resolve_options(o, N, lda, ldb);
    return plan_call(*st, M, N, K, static_cast<cudaStream_t>(stream_v), ro, st->ws_slots > 0, pl);
}

// ---------------------------------------------------------------------------
// the entry point that allocates nothing: stream-K scratch in a static array
// ---------------------------------------------------------------------------

// 20 MiB holds the stream-K workspace of the largest persistent grid on a
// 152-SM GB300 (76 pairs × 2 CTAs × 128 KiB of fp32 partials + flags).  Like
// every __device__ variable it is placed on each GPU that loads this library
// and kept there until the process exits.
constexpr size_t kStaticScratchBytes = size_t(20) << 20;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

struct StaticScratch {
    bool ready = false;
    bool ok = false;
    void* ptr = nullptr;   // device address of g_static_scratch on this device
};
StaticScratch g_static_scratch_addr[kMaxDevices];

// In host code `g_static_scratch` names a host-side stand-in, not device
// memory: the kernel must be given the address the runtime reports, looked up
// once per device with that device current.
gemm_status_t static_scratch(int dev, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    StaticScratch& sc = g_static_scratch_addr[dev];
    if (!sc.ready) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) cudaGetLastError();
        sc.ok = e == cudaSuccess && ptr != nullptr;
        sc.ptr = ptr;
        sc.ready = true;
    }
    if (!sc.ok) return GEMM_ERR_LAUNCH;
    *out = sc.ptr;
    return GEMM_OK;
}

gemm_status_t run_noalloc(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                          const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc, void* stream_v) {
    gemm_status_t s = check_args(M, N, K, A, lda, B, ldb, C, ldc);
    if (s != GEMM_OK) return s;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceState* st = nullptr;
    int dev = -1;
    if ((s = device_state(&st, &dev, false)) != GEMM_OK) return s;
#if G16_MCAST_LIB
    if ((s = check_local_operands(*st, dev, M, N, K, A, lda, B, ldb, false, false)) != GEMM_OK) return s;
#endif
    cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
    if (K == 0) return zero_fill(*st, M, N, C, ldc, stream);
    const gemm_f16_nt_options_t ro = resolve_options(nullptr, N, lda, ldb);
    gemm_f16_nt_plan_t pl;
    // As in gemm_f16_nt, a call made under stream capture is planned without
    // the stream-K split: a replay would repeat the launch id that tags the
    // split's completion flags in the shared scratch.
    if ((s = plan_call(*st, M, N, K, stream, ro, true, &pl)) != GEMM_OK) return s;
    void* ws = nullptr;
    if (pl.workspace_bytes > 0) {
        if (uint64_t(pl.workspace_bytes) > kStaticScratchBytes) return GEMM_ERR_SCRATCH_LIMIT;
        if ((s = static_scratch(dev, &ws)) != GEMM_OK) return s;
    }
    // Nothing in the scratch has to start at zero: each launch's completion
    // flags carry that launch's own 64-bit id, so values left by an earlier
    // call never match, and every partial tile is written before it is read.
    return launch_any(false, pl, M, N, K, A, lda, B, ldb, C, ldc, stream, &ro, st->watchdog, ws);
}

}  // namespace g16

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

G16_EXPORT gemm_status_t gemm_f16_nt(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                                     const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc,
                                     void* stream) {
    return g16::run(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr);
}

G16_EXPORT gemm_status_t gemm_f16_nt_noalloc(int64_t M, int64_t N, int64_t K, const uint16_t* A,
                                             int64_t lda, const uint16_t* B, int64_t ldb, uint16_t* C,
                                             int64_t ldc, void* stream) {
    return g16::run_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream);
}

G16_EXPORT gemm_status_t gemm_f16_nt_ex(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                                        const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc,
                                        void* stream, const gemm_f16_nt_options_t* opts) {
    return g16::run(M, N, K, A, lda, B, ldb, C, ldc, stream, opts);
}

G16_EXPORT gemm_status_t gemm_bf16_nt(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                                      const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc,
                                      void* stream) {
    return g16::run(M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr, true);
}

G16_EXPORT gemm_status_t gemm_bf16_nt_ex(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda,
                                         const uint16_t* B, int64_t ldb, uint16_t* C, int64_t ldc,
                                         void* stream, const gemm_f16_nt_options_t* opts) {
    return g16::run(M, N, K, A, lda, B, ldb, C, ldc, stream, opts, true);
}

G16_EXPORT gemm_status_t gemm_f16_nt_device_status(void* stream, uint32_t* flags) {
    g16::DeviceState* st = nullptr;
    gemm_status_t s = g16::current_device(&st);
    if (s != GEMM_OK) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    uint32_t v = 0;
    if (cudaMemcpy(&v, st->watchdog, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(st->watchdog, 0, sizeof(v)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    if (flags) *flags = v;
    return v ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

G16_EXPORT gemm_status_t gemm_f16_nt_device_limits(int32_t* sms, int32_t* resident_pairs,
                                                   int32_t* resident_ctas, int32_t* resident_pair_pairs) {
    g16::DeviceState* st = nullptr;
    gemm_status_t s = g16::current_device(&st);
    if (s != GEMM_OK) return s;
    if (sms) *sms = st->sms;
    if (resident_pairs) *resident_pairs = st->max_clusters2;
    if (resident_ctas) *resident_ctas = st->max_ctas1;
    if (resident_pair_pairs) *resident_pair_pairs = st->max_clusters4;
    return GEMM_OK;
}

G16_EXPORT gemm_status_t gemm_f16_nt_debug_status(void* stream) {
    return gemm_f16_nt_device_status(stream, nullptr);
}

G16_EXPORT gemm_status_t gemm_f16_nt_device_workspace(int32_t* slots, int64_t* bytes_per_slot) {
    g16::DeviceState* st = nullptr;
    gemm_status_t s = g16::current_device(&st);
    if (s != GEMM_OK) return s;
    if (slots) *slots = st->ws_slots;
    if (bytes_per_slot) *bytes_per_slot = st->ws_bytes;
    return GEMM_OK;
}

G16_EXPORT int32_t gemm_f16_nt_multicast_available(void) { return G16_MCAST_LIB ? 1 : 0; }

G16_EXPORT gemm_status_t gemm_f16_nt_launch_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                                 void* stream, const gemm_f16_nt_options_t* opts,
                                                 gemm_f16_nt_plan_t* plan) {
    return g16::launch_plan(M, N, K, lda, ldb, stream, opts, plan);
}

G16_EXPORT const char* gemm_f16_nt_status_string(gemm_status_t status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE: size or leading dimension out of range, or NULL pointer";
        case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED: pointers must be 16-byte aligned and leading dimensions multiples of 8";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "GEMM_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: a CUDA runtime or driver call failed";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a pipeline wait ran into the device watchdog";
        case GEMM_ERR_SCRATCH_LIMIT:
            return "GEMM_ERR_SCRATCH_LIMIT: the problem's stream-K scratch exceeds the 20 MiB static array "
                   "of gemm_f16_nt_noalloc; use gemm_f16_nt";
        case GEMM_ERR_NOT_LOCAL:
            return "GEMM_ERR_NOT_LOCAL: the multicast library takes only operands in device memory of the "
                   "current device, in a process that sees one GPU";
        default: return "unknown gemm_status_t";
    }
}

G16_EXPORT gemm_status_t gemm_f16_nt_plan(int64_t M, int64_t N, int64_t K, int32_t num_sms,
                                          int32_t max_clusters, const gemm_f16_nt_options_t* opts,
                                          gemm_f16_nt_plan_t* plan) {
    // the automatic choices as for contiguous operands (lda = ldb = K)
    const gemm_f16_nt_options_t ro = g16::resolve_options(opts, N, K, K);
    return g16::make_plan(M, N, K, num_sms, max_clusters, &ro, plan);
}

G16_EXPORT gemm_status_t gemm_f16_nt_tile_coord(int64_t linear, int32_t m_tiles, int32_t n_tiles,
                                                int32_t swizzle, int32_t* m_tile, int32_t* n_tile) {
    if (m_tiles < 1 || n_tiles < 1 || swizzle < 1 || swizzle > 64 || !m_tile || !n_tile)
        return GEMM_ERR_INVALID_VALUE;
    const int64_t total = int64_t(m_tiles) * n_tiles;
    const int64_t sw = swizzle < n_tiles ? swizzle : n_tiles;
    if (total >= (int64_t(1) << 31) || int64_t(m_tiles) * sw >= (int64_t(1) << 31) || linear < 0 ||
        linear >= total)
        return GEMM_ERR_INVALID_VALUE;
    g16::Raster r = g16::make_raster(uint32_t(m_tiles), uint32_t(n_tiles), uint32_t(swizzle));
    uint32_t m, n;
    g16::raster_coord(r, uint32_t(linear), m, n);
    *m_tile = int32_t(m);
    *n_tile = int32_t(n);
    return GEMM_OK;
}

G16_EXPORT gemm_status_t gemm_f16_nt_schedule(int64_t M, int64_t N, int64_t K, int32_t num_sms,
                                              int32_t max_clusters, const gemm_f16_nt_options_t* opts,
                                              int32_t cluster, gemm_f16_nt_item_t* items,
                                              int32_t max_items, int32_t* n_items) {
    if (!n_items || max_items < 0 || (max_items > 0 && !items)) return GEMM_ERR_INVALID_VALUE;
    gemm_f16_nt_plan_t pl;
    const gemm_status_t s = gemm_f16_nt_plan(M, N, K, num_sms, max_clusters, opts, &pl);
    if (s != GEMM_OK) return s;
    if (cluster < 0 || cluster >= pl.clusters) return GEMM_ERR_INVALID_VALUE;
    if (pl.kernel == 1) {
        // the small-problem kernel: cluster c computes piece c % s of tile c / s
        // (s = split_pieces, 1 without split-K); piece 0 owns the tile and adds
        // the others' partials, each piece covers an equal share of the k-blocks
        if (max_items > 0) {
            const int64_t np = pl.split_pieces, t = cluster / np, pc = cluster % np;
            gemm_f16_nt_item_t& o = items[0];
            memset(&o, 0, sizeof(o));
            o.tile = int32_t(t);
            o.m_tile = int32_t(t % pl.m_tiles);
            o.n_tile = int32_t(t / pl.m_tiles);
            o.kb0 = int32_t(pl.k_blocks * pc / np);
            o.kb1 = int32_t(pl.k_blocks * (pc + 1) / np);
            o.kind = np == 1 ? g16::kItemWhole : (pc == 0 ? g16::kItemOwner : g16::kItemPartialOut);
            o.partners = (np > 1 && pc == 0) ? int32_t(np - 1) : 0;
            o.parts = 1;
            o.pieces = 1;
        }
        *n_items = 1;
        return GEMM_OK;
    }
    // the launch's schedule fields, set exactly as the launch sets them
    struct {
        uint32_t num_tiles, num_kb, sk_tiles;
        uint64_t sk_units;
        uint32_t tail_first, tail_split, split_pieces, k_alternate, dyn_first;
    } sp;
    g16::set_schedule(sp, pl);
    const g16::Raster r = g16::make_raster(uint32_t(pl.m_tiles), uint32_t(pl.n_tiles), uint32_t(pl.swizzle));
    const uint32_t G = uint32_t(pl.clusters), c = uint32_t(cluster);
    g16::Work w;
    g16::Item it;
    g16::work_init(w, sp, c, G);
    int32_t n = 0;
    while (g16::work_next(w, sp, it)) {
        if (n < max_items) {
            gemm_f16_nt_item_t& o = items[n];
            uint32_t mt, nt;
            g16::raster_coord(r, it.tile, mt, nt);
            o.tile = int32_t(it.tile);
            o.m_tile = int32_t(mt);
            o.n_tile = int32_t(nt);
            o.kb0 = int32_t(it.kb0);
            o.kb1 = int32_t(it.kb1);
            o.kind = int32_t(it.kind);
            o.part = int32_t(it.part);
            o.parts = int32_t(it.parts);
            o.partners = it.kind == g16::kItemOwner ? int32_t(g16::owner_partners(sp, it.tile, c, G)) : 0;
            o.piece = int32_t(it.piece);
            o.pieces = int32_t(it.pieces);
            // the persistent kernel's producer order (an fp16 accumulator keeps k order)
            o.k_down = (opts && opts->accumulate == 1) ? 0 : int32_t(g16::item_k_down(sp, it, G));
        }
        ++n;
    }
    *n_items = n;
    return GEMM_OK;
}

G16_EXPORT gemm_status_t gemm_f16_nt_fast_divmod(uint32_t n, uint32_t d, uint32_t* q, uint32_t* r) {
    if (d < 1 || d > (1u << 31) || n >= (1u << 31) || !q || !r) return GEMM_ERR_INVALID_VALUE;
    g16::FastDiv f = g16::make_fastdiv(d);
    const uint32_t qq = g16::fastdiv_q(f, n);
    *q = qq;
    *r = n - qq * d;
    return GEMM_OK;
}
