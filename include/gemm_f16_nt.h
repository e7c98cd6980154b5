/*
 * gemm_f16_nt.h — C ABI of the GB300 (sm_103a) dense fp16 NT matrix multiply.
 *
 *     C[M,N] = A[M,K] · B[N,K]ᵀ      fp16 inputs, fp32 accumulation, fp16 output
 *
 * The operation is the one the Tilus "matmul-hopper" tutorial builds up in its
 * versions 2–6: A is an [m_size, k_size] fp16 matrix, B an [n_size, k_size]
 * fp16 matrix read transposed, the accumulator is fp32 and C is the fp16 cast
 * of it ("3. Warp Specialization", §The Full Kernel; "4. Pipeline Abstraction
 * and Two Consumer Warp Groups", §The Full Kernel; "6. Register Reallocation,
 * Multicast, and a Persistent Kernel", opening list: fp32 accumulation kept).
 * The tutorial's kernels take three sizes and three contiguous pointers; this
 * ABI adds leading dimensions and a stream.
 *
 * Numbers: fp16 values are IEEE-754 binary16 bit patterns (uint16_t).  The sum
 * over k is carried in fp32 on the tensor cores; the fp32 → fp16 cast rounds to
 * nearest, ties to even, overflowing to ±inf.  Results agree with an fp64
 * reference rounded once to fp16 within 2 fp16 ulps + 1e-4·sqrt(K) per
 * element, and exactly when every partial sum is an fp32-exact integer.
 *
 * Threading: every entry point may be called from any host thread.  Each GEMM
 * call is asynchronous on the given stream.
 *
 * Two kernels.  The persistent kernel (256×256 tiles on CTA pairs, one
 * persistent cluster per pair of SMs, a work schedule with stream-K, N-split
 * and split pieces) computes every problem whose 128-row tiles would not fit
 * on the SMs in one wave.  The small-problem kernel computes one 128×tile_n
 * tile (tile_n = 32, 64 or 128, the narrowest whose tiles fit on the SMs at
 * once) per CTA, for problems whose tiles do fit: there the persistent
 * kernel's 256×256 tiles would leave most SMs idle and its fixed costs
 * dominate.  With few tiles and k of at least 2048 (32 k-blocks) it cuts each
 * tile along k into up to 8 pieces on their own CTAs (split-K, at least 8
 * k-blocks a piece, all in one wave); the first piece owns the tile and adds
 * the others' fp32 partials, which they pass through the workspace, in k
 * order, so results do not depend on timing.  It takes problems with at most
 * 128 k-blocks a piece.  The automatic choice applies when no persistent-
 * kernel option is given (see gemm_f16_nt_ex); gemm_f16_nt_launch_plan reports
 * which kernel a call gets (plan field `kernel`).  Both give results within the
 * same bound; only the order of the fp32 additions can differ between them.
 *
 * Two builds share this header.  libgemm_f16_nt.so is the library; it issues
 * no multicast copy and may be loaded by each of several processes on several
 * GPUs.  libgemm_f16_nt_mcast.so, built only on request, is the same library
 * plus clusters of two CTA pairs that share A by TMA multicast (cluster_pairs
 * below); it is for single-GPU processes and refuses any other use
 * (GEMM_ERR_NOT_LOCAL).
 */
#ifndef GEMM_F16_NT_H_
#define GEMM_F16_NT_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,      /* a size or leading dimension is out of range, or a pointer is NULL */
    GEMM_ERR_MISALIGNED = 2,         /* a pointer or row pitch breaks the 16-byte rule below */
    GEMM_ERR_UNSUPPORTED_DEVICE = 3, /* no CUDA device, or the current device is not compute capability 10.3 */
    GEMM_ERR_LAUNCH = 4,             /* the CUDA runtime or driver refused a call (set-up or launch) */
    GEMM_ERR_TIMEOUT = 5,            /* the device watchdog word is set (see gemm_f16_nt_device_status) */
    GEMM_ERR_SCRATCH_LIMIT = 6,      /* gemm_f16_nt_noalloc: the scratch needed exceeds its static array */
    GEMM_ERR_NOT_LOCAL = 7           /* multicast library only: an operand is not device memory of the
                                        current device, or the process sees more than one GPU */
} gemm_status_t;

/*
 * gemm_f16_nt — C = A · Bᵀ on the current CUDA device.
 *
 *   M, N, K   sizes, each in [0, 2^31).
 *   A         device pointer, element (m, k) at A[m*lda + k], m < M, k < K.
 *   lda       row pitch of A in elements, lda >= max(K, 1).
 *   B         device pointer, element (n, k) at B[n*ldb + k], n < N, k < K.
 *   ldb       row pitch of B in elements, ldb >= max(K, 1).
 *   C         device pointer, element (m, n) at C[m*ldc + n], m < M, n < N.
 *   ldc       row pitch of C in elements, ldc >= max(N, 1).
 *   stream    a cudaStream_t (NULL = the legacy default stream).
 *
 * Layout and alignment: all three matrices are row-major.  A, B and C must be
 * 16-byte aligned and lda, ldb, ldc multiples of 8 elements (16 bytes): the
 * tensor-memory-accelerator copies that move the tiles require it.  There is
 * no slower path for other layouts: such calls return GEMM_ERR_MISALIGNED.
 *
 * Semantics: C is overwritten (no alpha/beta).  Only the M×N window is
 * written; columns N..ldc-1 of each row of C are never touched.  M == 0 or
 * N == 0 is a no-op.  K == 0 writes +0 to the whole M×N window (the empty sum).
 * C must not overlap A or B (not checked).
 *
 * Ownership: the caller owns A, B and C and keeps them alive until the work on
 * `stream` completes.  The library keeps no pointer after the call returns,
 * and allocates nothing per call.  The first call on a device performs
 * one-time set-up on that device: device query, kernel attributes, the
 * watchdog word's address, and the reservation (cudaMalloc) of the stream-K
 * workspace, GEMM_F16_NT_WORKSPACE_SLOTS slots (environment variable, 0..8,
 * default 4) of about 20 MB each on a 152-SM GPU, kept until the process exits
 * (gemm_f16_nt_device_workspace reports them).  Shapes whose last wave of
 * output tiles would leave enough SMs idle use a stream-K schedule (see
 * `schedule` below) that takes one slot, round-robin.  Before such a launch
 * the call makes `stream` wait for the previous launch that used the same slot
 * (cudaStreamWaitEvent on an event the call records after each launch), so
 * calls on unordered streams never use one slot at the same time: up to that
 * many stream-K calls run concurrently, and more are ordered.  If the
 * reservation fails, or the environment variable is 0, every call is planned
 * without the split; gemm_f16_nt_launch_plan reports it (split_k_off = 2).
 *
 * Ordering: the kernel is launched with programmatic stream serialization, so
 * its CTAs may start their set-up (shared memory, barriers, tensor memory)
 * while the kernel before it on `stream` is still draining.  It reads and
 * writes no global memory (A, B, C, workspace, watchdog word) until that
 * kernel has completed and its writes are visible (griddepcontrol.wait), so
 * stream order holds as for any other launch.
 *
 * Stream capture: a call made while `stream` is being captured into a CUDA
 * graph is planned without the stream-K split (schedule 2 included), because
 * a replay repeats the launch's parameters and the split's completion flags
 * are tagged per launch (split_k_off = 1 in gemm_f16_nt_launch_plan); for the
 * same reason its last wave is dealt round-robin, not claimed.  The
 * captured kernel then touches only A, B, C, the watchdog word and (if
 * requested) the trace buffer, so the graph can be replayed any number of
 * times.  Make the first call on a device outside any capture: it sets the
 * device up (kernel attributes, the workspace reservation).
 *
 * Errors: invalid arguments are reported before anything is enqueued, and C is
 * left unchanged.  The call returns after enqueueing; a fault during execution
 * surfaces at the caller's next synchronisation, and a watchdog expiry (a
 * pipeline wait that did not finish within the time limit) sets the device
 * watchdog word read by gemm_f16_nt_device_status.
 */
gemm_status_t gemm_f16_nt(int64_t M, int64_t N, int64_t K,
                          const uint16_t *A, int64_t lda,
                          const uint16_t *B, int64_t ldb,
                          uint16_t *C, int64_t ldc,
                          void *stream);

/*
 * gemm_f16_nt_noalloc — gemm_f16_nt for callers that cannot allocate device
 * memory during the call.
 *
 * No counterpart in the tutorial pages: this is an interface choice of the
 * library, not part of the method.
 *
 * Who needs it: gemm_f16_nt reserves its stream-K workspace (four slots of
 * about 20 MB) with cudaMalloc on its first call on a device.  Some callers
 * cannot let a library allocate at all, not even once: processes whose device
 * memory is reserved up front by their own allocator, so that an extra
 * allocation can fail or fragment it, and latency-critical loops whose first
 * call must not pay an allocation's cost or implicit synchronisation.
 * This entry point computes the same product with the same kernel and the same
 * schedule, and takes no memory at all during the call: its scratch is a
 * fixed array of 20 MiB (20,971,520 bytes) compiled into the library, which
 * every GPU that loads the library holds until the process exits.
 *
 * Arguments, layout, alignment, ownership and errors are those of gemm_f16_nt.
 * Extra rules:
 *   - It calls no cudaMalloc, cudaFree, pool or other allocating routine.
 *   - Its first call on a device also looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); later calls reuse it.
 *   - Every call on a device shares the one array, which keeps what the last
 *     call left in it.  Calls that can overlap on the GPU (for example on two
 *     streams with no ordering between them) race on it and may return wrong
 *     results: order them, e.g. keep them on one stream.  Nothing in the array
 *     has to start at zero (each launch tags its completion flags with its own
 *     id, and writes every partial tile before reading it).
 *   - A problem whose stream-K scratch would exceed the array (possible only
 *     on GPUs with more than 152 SMs) is rejected with GEMM_ERR_SCRATCH_LIMIT
 *     before anything is enqueued.
 *   - Like gemm_f16_nt, a call made while `stream` is capturing is planned
 *     without the stream-K split, so it does not use the array.
 */
gemm_status_t gemm_f16_nt_noalloc(int64_t M, int64_t N, int64_t K,
                                  const uint16_t *A, int64_t lda,
                                  const uint16_t *B, int64_t ldb,
                                  uint16_t *C, int64_t ldc,
                                  void *stream);

/*
 * Tuning and test options for gemm_f16_nt_ex.  Zero (or NULL) in any field
 * selects the default that gemm_f16_nt uses.
 *
 *   cta_group     2: a CTA pair computes one 256×256 tile with 2-SM MMAs and
 *                 each CTA loads half of the shared B tile (the persistent
 *                 kernel's default); 1: one CTA computes a 128×256 tile on
 *                 its own.  0 (automatic): the small-problem kernel where it
 *                 applies (one CTA per tile), else 2.  A nonzero value selects
 *                 the persistent kernel unless schedule is 5, where it is the
 *                 small-problem kernel's CTA group (2: 256×tile_n tiles on a
 *                 CTA pair, each CTA loading tile_n/2 rows of B).
 *   swizzle       width, in N tiles, of the groups of the tile raster; tiles
 *                 in a group are visited row-major so that concurrently
 *                 running tiles share B columns in L2 (Tilus tutorial
 *                 "4. Pipeline Abstraction and Two Consumer Warp Groups",
 *                 §Tile Rasterization), odd groups from the last row up
 *                 (see gemm_f16_nt_tile_coord).  Range 1..64; default 8.
 *   max_clusters  upper bound on the persistent grid, in CTA pairs (or CTAs
 *                 for cta_group 1); 0 = as many as can be resident.
 *   timeout_ns    watchdog limit, in ns, for a wait on one pipeline stage
 *                 (default 1 s).  Waits that can last a whole work item (the
 *                 epilogue's wait for a finished accumulator, a stream-K
 *                 owner's wait for its partners' partial tiles, the MMA
 *                 issuer's wait for a drained accumulator and the producer's
 *                 wait for a free stage behind it) get timeout_ns plus 8 us
 *                 per 64-wide k-block of K, so that deep-K problems finish:
 *                 K = 2^30 allows each of them about 134 s.
 *   inject_stall  test hook: if nonzero the TMA producers issue nothing, so
 *                 every consumer wait runs into the watchdog; the kernel then
 *                 sets the watchdog word, releases its tensor memory and
 *                 exits without writing C.
 *   schedule      0 (default): whole tiles round-robin over the persistent
 *                 clusters, except that when at least 8 % of that schedule's
 *                 tile slots would sit idle in its last wave (one pair per
 *                 cluster), the k-block work of the last wave plus one full
 *                 wave is split evenly across all clusters (stream-K), with
 *                 fp32 partial tiles summed by each tile's first piece in a
 *                 fixed order (results are reproducible run to run).  The
 *                 last-wave split needs deep k (at least 32 k-blocks spared a
 *                 cluster) and at least one full wave of whole tiles beside it.
 *                 With fewer tiles than clusters and k of at least 48 k-blocks
 *                 (64 k each), every tile is cut along k into s = 2, 4 or 8
 *                 equal split pieces (the largest with tiles·s <= clusters, at
 *                 least 2 k-blocks a piece) on their own clusters; the tile's
 *                 columns are cut into s slices, and each piece writes the
 *                 fp32 partials of the other pieces' slices, then sums the s
 *                 partials of its own slice in piece (k) order and stores it.
 *                 With fewer tiles than clusters and shallower k, the N-split
 *                 below applies;
 *                 1: whole tiles only; 2: stream-K whenever possible (tests;
 *                 with fewer tiles than clusters, all their k-blocks spread
 *                 over the clusters, owners adding their partners'
 *                 partials); 3: N-split whenever possible (tests); 4: split
 *                 pieces whenever there is room for two a tile (tests; pieces
 *                 of one k-block allowed); 5: the small-problem kernel for any
 *                 problem (K-major A and B, fp32 accumulator, one pair per
 *                 cluster, no trace; GEMM_ERR_INVALID_VALUE otherwise).
 *                 The automatic plan (schedule 0 with cta_group, swizzle,
 *                 max_clusters and tile_n 0, cluster_pairs at most 1) takes the
 *                 small-problem kernel when those conditions hold, its 128×32,
 *                 128×64 or 128×128 tiles fit on the device's SMs in one wave
 *                 and each CTA's k range (after its split-K, if any) is at
 *                 most 128 k-blocks.  Its split-K, like stream-K, needs a
 *                 workspace slot and is off under stream capture.
 *                 N-split: when the stream-K rule does not split the problem
 *                 and either there are fewer tiles than clusters or k is
 *                 shallow (at most 32 k-blocks), the R tiles of the last wave
 *                 (all tiles, with fewer tiles than clusters) are each cut
 *                 along N into s = 2 or 4 narrower tiles (256×128 or 256×64, s
 *                 the largest with R·s <= clusters) that run on their own CTA
 *                 pairs; nothing is summed across clusters.
 *                 A narrower MMA is not proportionally faster on these tensor
 *                 cores (with no loads, N = 128 takes 69 % and N = 64 62 % of
 *                 the 256-wide time per k-block), and with their operand loads
 *                 the slices measured no faster than whole tiles, so this
 *                 mainly shortens each cluster's epilogue: it is for small,
 *                 latency-bound problems.
 *                 With 3 the last R tiles of any problem are cut the same way
 *                 when 2R <= clusters.  N-split and split pieces need one CTA
 *                 pair per cluster; the N-split also B stored [N, K].  An fp16
 *                 accumulator never splits in k.
 *                 A stream-K or split-piece launch needs a workspace
 *                 (gemm_f16_nt_plan's workspace_bytes): one of the slots
 *                 reserved at the device's set-up (see Ownership above).
 *                 Without slots, or under stream capture, the call is planned
 *                 as with schedule 0 but with no split in k, neither stream-K
 *                 nor split pieces (plan field split_k_off).
 *   trace, trace_items
 *                 debugging aid: if `trace` is a device pointer to
 *                 clusters × trace_items × 8 uint64 (zeroed by the caller), the
 *                 kernel records for each work item i < trace_items of each
 *                 cluster c, at trace[(c·trace_items + i)·8 + j]:
 *                 j=0 tile | kind << 32 (0 whole, 1 partial piece, 2 owner),
 *                 j=1 kb0 | kb1 << 32, and %globaltimer stamps (ns) j=2 MMA
 *                 issue start, j=3 MMA issue end, j=4 accumulator ready at the
 *                 epilogue, j=5 partner partials ready, j=6 epilogue done
 *                 (stamps from the leader CTA's MMA thread and one of its
 *                 epilogue warps), j=7 total ns the MMA thread waited for
 *                 filled pipeline stages during the item.
 *   cluster_pairs 1: a cluster is one CTA pair; 2 (multicast library only;
 *                 GEMM_ERR_INVALID_VALUE in libgemm_f16_nt.so): a cluster is
 *                 two CTA pairs side by side in N (a 256×512 tile) that share
 *                 their A rows: each CTA loads half of its A tile and TMA
 *                 multicasts it to the same-rank CTA of the other pair, which
 *                 halves A's L2 → SM traffic.  Clusters of four CTAs fit on
 *                 fewer SMs (144 of 152 on a GB300).  Needs cta_group 2.
 *                 Default (0): 1 in libgemm_f16_nt.so; in the multicast
 *                 library 2 when lda or ldb is not a multiple of 64 elements
 *                 (128 bytes: each 128-byte row slice of a tile then spans two
 *                 L2 lines and L2 traffic is the limit) and N > 256, else 1.
 *   a_layout      0 (default): A is stored [M, K], element (m, k) at
 *                 A[m*lda + k]; 1: A is stored [K, M] (M contiguous), element
 *                 (m, k) at A[k*lda + m], lda >= M.
 *   b_layout      0 (default): B is stored [N, K], element (n, k) at
 *                 B[n*ldb + k]; 1: B is stored [K, N], element (n, k) at
 *                 B[k*ldb + n], ldb >= N.
 *                 The product is always C[M,N] = Σ_k A(m,k)·B(n,k) with C
 *                 row-major: layouts (0,1) give C = A·B for a row-major [K, N]
 *                 B, (1,0) give C = Aᵀ·Bᵀ-style transposed storage, etc.  The
 *                 tensor cores read M/N-contiguous tiles as MN-major operands.
 *   tile_n        the small-problem kernel's tile width: 32, 64 or 128
 *                 columns; 0 (default) = the narrowest whose tiles fit on the
 *                 SMs in one wave (128 if none does).  Any other value returns
 *                 GEMM_ERR_INVALID_VALUE; a nonzero value keeps the automatic
 *                 plan on the persistent kernel (use it with schedule 5).
 *   accumulate    0 (default): fp32 accumulator, rounded once to fp16 at the
 *                 end (the method as the tutorial pages define it);
 *                 1: fp16 accumulator (fp16 operands only: gemm_f16_nt_ex).
 *                 The tensor cores add each 16-wide k step to an fp16
 *                 accumulator, so the result carries one fp16 rounding per 16
 *                 k instead of one in all.  This is the variant the pages set
 *                 against fp32 accumulation ("6. Register Reallocation,
 *                 Multicast, and a Persistent Kernel", §Shared-Memory
 *                 Epilogue, the Note on an earlier version: over K = 8192 with
 *                 unit-variance outputs, mean absolute error 0.0023 against
 *                 0.00014, maximum 0.047).  It runs whole tiles only (no
 *                 stream-K split).  On these tensor cores the fp16 accumulator
 *                 takes the same tensor-memory columns as fp32 (one value per
 *                 32-bit column), so the tile shapes are the same.  Any other value, or 1 with bf16 operands, returns
 *                 GEMM_ERR_INVALID_VALUE.
 */
typedef struct {
    int32_t cta_group;
    int32_t swizzle;
    int32_t max_clusters;
    int32_t inject_stall;
    uint64_t timeout_ns;
    int32_t schedule;
    int32_t trace_items;
    uint64_t *trace;
    int32_t cluster_pairs;
    int32_t a_layout;
    int32_t b_layout;
    int32_t accumulate;
    int32_t tile_n;
} gemm_f16_nt_options_t;

/* gemm_f16_nt with options (opts may be NULL).  Same arguments, layout,
 * ownership and errors as gemm_f16_nt; an option out of range returns
 * GEMM_ERR_INVALID_VALUE. */
gemm_status_t gemm_f16_nt_ex(int64_t M, int64_t N, int64_t K,
                             const uint16_t *A, int64_t lda,
                             const uint16_t *B, int64_t ldb,
                             uint16_t *C, int64_t ldc,
                             void *stream, const gemm_f16_nt_options_t *opts);

/*
 * gemm_bf16_nt, gemm_bf16_nt_ex — the same product with bfloat16 operands and
 * result: C[M,N] = A[M,K] · B[N,K]ᵀ, bf16 in, fp32 accumulation, bf16 out.
 *
 * The tutorial pages compute in fp16 only; bf16 is this library's variant of
 * the same method (same kernel, schedule and options; the tensor cores read
 * bf16 operands and the epilogue rounds the fp32 accumulator to the nearest
 * bf16, ties to even).  A, B and C hold bf16 bit patterns (1 sign, 8 exponent,
 * 7 fraction bits).  Arguments, layout, alignment, ownership, options and
 * errors are those of gemm_f16_nt / gemm_f16_nt_ex.  Results agree with an
 * fp64 reference rounded once to bf16 within 2 bf16 ulps + 1e-4·sqrt(K), and
 * exactly when every partial sum is an fp32-exact integer.
 */
gemm_status_t gemm_bf16_nt(int64_t M, int64_t N, int64_t K,
                           const uint16_t *A, int64_t lda,
                           const uint16_t *B, int64_t ldb,
                           uint16_t *C, int64_t ldc,
                           void *stream);
gemm_status_t gemm_bf16_nt_ex(int64_t M, int64_t N, int64_t K,
                              const uint16_t *A, int64_t lda,
                              const uint16_t *B, int64_t ldb,
                              uint16_t *C, int64_t ldc,
                              void *stream, const gemm_f16_nt_options_t *opts);

/*
 * gemm_f16_nt_device_status — read and clear the current device's watchdog word.
 *
 * Synchronises `stream`, copies the word into *flags (may be NULL) and resets
 * it to 0.  Returns GEMM_ERR_TIMEOUT if it was nonzero, GEMM_OK if it was 0,
 * GEMM_ERR_LAUNCH if the synchronisation or copy failed (for example after an
 * earlier fault), GEMM_ERR_UNSUPPORTED_DEVICE without a usable device.
 * Bit 0 of the word: a wait expired.  Bit 7+s: wait site s expired, with
 * s = 1 producer waiting for a free ring slot, 2 MMA issuer waiting for a
 * filled slot, 3 MMA issuer waiting for a free accumulator, 4 epilogue waiting
 * for a finished accumulator, 5 producer teardown waiting for its copies,
 * 6 MMA teardown waiting for its MMAs, 7 a stream-K owner waiting for a
 * partner's partial tile, 8 a role waiting for its cluster's claim of a
 * last-wave tile (or the claim itself failing).  The word is shared by every
 * call on that device.
 */
gemm_status_t gemm_f16_nt_device_status(void *stream, uint32_t *flags);

/* gemm_f16_nt_device_status(stream, NULL): GEMM_OK if no wait expired since
 * the word was last read, GEMM_ERR_TIMEOUT if one did (the word is cleared). */
gemm_status_t gemm_f16_nt_debug_status(void *stream);

/* The stream-K workspace reserved on the current device at its set-up: the
 * number of slots (0: the split is off for every call) and the bytes of each.
 * Either pointer may be NULL. */
gemm_status_t gemm_f16_nt_device_workspace(int32_t *slots, int64_t *bytes_per_slot);

/* 1 in the multicast library (libgemm_f16_nt_mcast.so), 0 in libgemm_f16_nt.so. */
int32_t gemm_f16_nt_multicast_available(void);

/*
 * What the one-time set-up found on the current device: its SM count and how
 * many clusters of the GEMM kernel can be resident at once (the persistent
 * grid sizes): CTA pairs (cta_group 2), single CTAs (cta_group 1), and
 * clusters of two pairs (cluster_pairs 2; 0 in libgemm_f16_nt.so, which has
 * no such configuration).  Any pointer may be NULL.
 * GEMM_ERR_UNSUPPORTED_DEVICE without a usable device.
 */
gemm_status_t gemm_f16_nt_device_limits(int32_t *sms, int32_t *resident_pairs,
                                        int32_t *resident_ctas, int32_t *resident_pair_pairs);

/* A static, human-readable name for a gemm_status_t value. */
const char *gemm_f16_nt_status_string(gemm_status_t status);

/* ---- host-only helpers (no CUDA call; used by the scheduler and its tests) ---- */

/*
 * The launch plan gemm_f16_nt would use for a problem with contiguous operands
 * (lda = ldb = K; the automatic cluster choice depends on them) on a device
 * with `num_sms` SMs and room for `max_clusters` resident clusters of the
 * chosen kind (0 = num_sms divided by the CTAs per cluster).  Returns
 * GEMM_ERR_INVALID_VALUE for sizes or options out of range.
 */
typedef struct {
    int32_t cta_group;     /* 1 or 2 */
    int32_t tile_m;        /* rows of C per cluster tile (128 · cta_group) */
    int32_t tile_n;        /* columns of C per cluster tile */
    int32_t block_k;       /* k per pipeline stage */
    int32_t stages;        /* shared-memory ring depth */
    int32_t m_tiles;       /* cdiv(M, tile_m) */
    int32_t n_tiles;       /* cdiv(N, tile_n) */
    int32_t k_blocks;      /* cdiv(K, block_k) */
    int64_t num_tiles;     /* m_tiles · n_tiles */
    int32_t clusters;      /* persistent clusters launched */
    int32_t grid_ctas;     /* clusters · cta_group · cluster_pairs */
    int32_t swizzle;       /* raster group width actually used */
    int32_t smem_bytes;    /* dynamic shared memory per CTA */
    int32_t tmem_cols;     /* tensor-memory columns allocated per CTA */
    int32_t sk_tiles;      /* tiles [0, sk_tiles) are split in k across all clusters (stream-K) */
    int32_t cluster_pairs; /* CTA pairs per cluster (tile_n = 256 · cluster_pairs) */
    int64_t workspace_bytes; /* device workspace a stream-K launch needs (0 if none) */
    int32_t tail_tiles;    /* the last tail_tiles tiles are each split in N (N-split) ... */
    int32_t tail_split;    /* ... into tail_split narrower tiles (1 = no split) */
    int32_t split_k_off;   /* gemm_f16_nt_launch_plan only: 0, or why the shape's stream-K
                              split is not taken: 1 the stream is capturing, 2 no workspace
                              was reserved on the device */
    int32_t split_pieces;  /* > 1: every tile is cut along k into split_pieces equal pieces,
                              one per cluster (clusters = num_tiles · split_pieces);
                              the persistent kernel's pieces reduce each other's fp32
                              partials, the small-problem kernel's first piece adds
                              the others'; 1 = not used */
    int32_t kernel;        /* 0: the persistent kernel; 1: the small-problem kernel: one
                              tile_m × tile_n tile per cluster (CTA or CTA pair), or
                              with split_pieces = s > 1 one of s k-pieces of it:
                              clusters = num_tiles · s, cluster c on piece c % s of
                              tile t = c / s at m_tile = t % m_tiles, n_tile =
                              t / m_tiles; piece 0 owns the tile (schedule kind 2) */
    int32_t k_order;       /* persistent kernel, fp32 accumulator: 1 when whole tiles of
                              odd rounds (round = (tile - sk_tiles) / clusters) load
                              their k-blocks from the last one down, so that a round
                              starts on the k-slabs the one before read last (taken
                              when one round's A and B strips, about
                              (clusters/swizzle + swizzle) strips of 256 rows × K,
                              exceed 60 MB); 0: every whole tile from k-block 0 up.
                              The k order of a sum changes only its rounding. */
    int32_t claimed_tiles; /* persistent kernel, whole tiles: the tiles of a last,
                              partial wave (num_tiles - claimed_tiles onward), which
                              are not dealt round-robin: each cluster, once it has
                              run its share, claims one of them at run time (a
                              launch-tagged counter in device memory), so that the
                              clusters that finish first take them.  0: every tile
                              dealt round-robin (stream-K, N-split, split pieces, a
                              single wave, or a call under stream capture).  The
                              schedule helper lists them as if cluster c took the
                              c-th. */
} gemm_f16_nt_plan_t;

gemm_status_t gemm_f16_nt_plan(int64_t M, int64_t N, int64_t K, int32_t num_sms,
                               int32_t max_clusters,
                               const gemm_f16_nt_options_t *opts,
                               gemm_f16_nt_plan_t *plan);

/*
 * The plan gemm_f16_nt_ex(M, N, K, A, lda, B, ldb, …, stream, opts) would
 * launch on the current device right now: the device's SM count and resident
 * clusters, the automatic choices for these leading dimensions, and the
 * split's availability (stream capture, reserved workspace; see split_k_off).
 * Performs the device's one-time set-up if it has not happened yet.  Errors
 * as gemm_f16_nt_plan, plus GEMM_ERR_UNSUPPORTED_DEVICE and GEMM_ERR_LAUNCH.
 */
gemm_status_t gemm_f16_nt_launch_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                      void *stream, const gemm_f16_nt_options_t *opts,
                                      gemm_f16_nt_plan_t *plan);

/*
 * One work item of the persistent schedule (gemm_f16_nt_schedule).
 */
typedef struct {
    int32_t tile;       /* linear index in the tile raster */
    int32_t m_tile;     /* its coordinates (gemm_f16_nt_tile_coord); with two */
    int32_t n_tile;     /*   CTA pairs per cluster, in 256×512 cluster tiles  */
    int32_t kb0, kb1;   /* k-block range [kb0, kb1), 64 k per block           */
    int32_t kind;       /* 0: whole k range; 1: stream-K piece that does not
                           start at k-block 0 (written as an fp32 partial tile
                           to the cluster's workspace slot); 2: stream-K piece
                           from k-block 0 that ends early (the tile's owner:
                           adds the partners' partials and stores C); 3: one
                           of split_pieces equal pieces of the tile (writes the
                           partial of the column slices it does not own, adds
                           the others' partials of the slices it owns)        */
    int32_t part;       /* column slice `part` of `parts` (N-split);          */
    int32_t parts;      /*   parts = 1: the whole tile width                  */
    int32_t partners;   /* kind 2: the number of following clusters whose
                           partial pieces it adds, in cluster order; else 0   */
    int32_t piece;      /* kind 3 (split piece): its index in the tile's      */
    int32_t pieces;     /*   pieces, 0 <= piece < pieces; else 0 and 1        */
    int32_t k_down;     /* 1: the item's k-blocks are loaded from kb1 - 1 down
                           to kb0 (kind 1, and kind 0 in odd rounds with
                           plan.k_order = 1); 0: from kb0 up                  */
} gemm_f16_nt_item_t;

/*
 * gemm_f16_nt_schedule — the work items, in order, that persistent cluster
 * `cluster` of the launch gemm_f16_nt_ex(M, N, K, …, opts) would run on a GPU
 * with `num_sms` SMs and at most `max_clusters` resident clusters (0: as many
 * as fit), from the same plan (gemm_f16_nt_plan) and the same schedule code
 * the kernel runs.  For a plan on the small-problem kernel (kernel = 1) each
 * cluster has one item: tile `cluster`, all of k.  Host only, for tests and
 * tools; no GPU is needed.
 *   items      caller-owned array of max_items entries (may be NULL if 0);
 *              the first min(n, max_items) items are written.
 *   n_items    receives n, the cluster's total number of items.
 * Returns GEMM_ERR_INVALID_VALUE for a bad argument or a cluster outside
 * [0, plan.clusters), and the plan's error for an invalid problem.
 */
gemm_status_t gemm_f16_nt_schedule(int64_t M, int64_t N, int64_t K, int32_t num_sms,
                                   int32_t max_clusters, const gemm_f16_nt_options_t *opts,
                                   int32_t cluster, gemm_f16_nt_item_t *items, int32_t max_items,
                                   int32_t *n_items);

/*
 * The tile raster: linear tile index -> (m_tile, n_tile).  N tiles are taken
 * in groups of `swizzle` columns (the last group may be narrower); inside a
 * group tiles go row-major (Tilus tutorial "4. Pipeline Abstraction and Two
 * Consumer Warp Groups", §Tile Rasterization), with rows taken in reverse in
 * odd groups, so that each group starts on the row strips where the one
 * before it ended.  A bijection of [0, m_tiles·n_tiles) onto the grid.  This
 * is the same function the kernel runs.
 */
gemm_status_t gemm_f16_nt_tile_coord(int64_t linear, int32_t m_tiles, int32_t n_tiles,
                                     int32_t swizzle, int32_t *m_tile, int32_t *n_tile);

/*
 * The multiply-shift division the kernel uses for divisors fixed per launch
 * (Granlund & Montgomery, "Division by Invariant Integers using
 * Multiplication", 1994, round-up variant): quotient and remainder of n / d for
 * 0 <= n < 2^31, 1 <= d < 2^31.
 */
gemm_status_t gemm_f16_nt_fast_divmod(uint32_t n, uint32_t d, uint32_t *q, uint32_t *r);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_F16_NT_H_ */
