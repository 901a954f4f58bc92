/*
 * ringattn.h — C ABI of libringattn.so: the single-GPU hot path of Ring Attention
 * (online-softmax merge over P virtual KV shards) for NVIDIA GB300 (sm_103a).
 *
 * The method. Queries of virtual device u stay put; at ring step s = 0..P-1 the
 * device scores them against the circulating key/value shard b = (u - s) mod P,
 *     S = Q_u K_b^T / sqrt(d_h),
 * and folds S into a running accumulator (m, z, y) — running row max, running
 * denominator, running unnormalised output — with the exact rescale
 * alpha = exp(m_old - m_new); after all P shards O = y / z.
 *   Source: "Ring Attention" (aarnphm.xyz, thoughts/ring-attention), the ring
 *   recurrence display; the same update as "Building block: the online-softmax
 *   trick" in "Ring Attention: Distributed Attention Across Devices"
 *   (aicomputerinstitute chapter) and §4.4 "Online Softmax Across KV Blocks" of
 *   "Part 4: Ring Attention" (Fofadiya).
 * On one GPU the P devices are virtual: a shard is an index range of tensors
 * that all sit in this GPU's memory, and "receiving" a shard is loading its tiles.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Tensors are in ORIGINAL token order whatever the shard layout (the layout is
 *  an index map, not a permutation of memory):
 *    q           [B, N, H, d]  bf16, row-major (d fastest)
 *    o           [B, N, H, d]  bf16, or fp32 when p->o_dtype == RA_DTYPE_F32
 *    k, v        [B, N, G, d]  bf16
 *    lse, m, z   [B, H, N]     fp32
 *    y           [B, N, H, d]  fp32
 *  B = batch, N = seqlen, H = heads, G = kv_heads (H % G == 0; query head h
 *  reads kv head floor(h*G/H)), d = head_dim in {64, 128}.
 *  LSE = m + ln z (natural log of the scaled scores); a row that admitted no
 *  key has O = 0 and LSE = -inf.
 *  Causal masking is on global positions: query token t sees key tokens <= t
 *  ("Ring Attention: what the near-infinite context paper actually says",
 *  "The causal masking complication").
 *
 *  Pointers named q,k,v,o,lse,m,z,y,o_parts,lse_parts,dout,dq,dk,dv,workspace
 *  are DEVICE pointers, allocated and owned by the caller, 16-byte aligned —
 *  except the host pointers of ring_attn_fwd_host and of the host shard map,
 *  which say so. The library allocates no device memory; its static device
 *  memory is one status word per GPU and the fixed scratch array of
 *  ring_attn_decode_noalloc. `stream` is a cudaStream_t (NULL = legacy default
 *  stream); every call that takes one is asynchronous on it. Calls on one
 *  stream are ordered; the library holds no per-call host state beyond the
 *  ordering events and copy streams that ring_attn_fwd_host creates and releases
 *  itself, so
 *  concurrent calls on different streams are safe when their output buffers
 *  (and workspaces) do not overlap.
 *
 *  CUDA graphs: after the first eager call of an entry point in a device's
 *  context (which sets the kernels' shared-memory limits and reads the device's
 *  facts; a context made anew, e.g. after cudaDeviceReset, gets the same first
 *  step at its first call, since the library keys these facts by context), the calls
 *  that launch kernels on `stream` only — every one but ring_attn_fwd_host and
 *  ring_attn_last_error — may be captured into a graph; a replay computes what
 *  the eager call would on the buffers' contents at replay time.
 *
 *  Outputs, in/out state and workspaces must not overlap one another or any
 *  input (inputs may overlap each other, e.g. the same tensor passed as k and
 *  v): a call whose written ranges would share a byte with another argument's
 *  range, counted from the shapes above, returns RA_ERR_INVALID_ARG. There is no
 *  in-place form.
 *
 *  Errors: argument errors are returned synchronously before any launch and
 *  nothing is written. Every device pointer is checked to be memory the current
 *  device's kernels may touch (its device memory — cudaMalloc, pools, virtual-memory
 *  mappings — or managed memory); host memory and other devices' memory give
 *  RA_ERR_INVALID_ARG instead of a kernel that would fault. RA_ERR_CUDA means a CUDA call (launch or tensor-map
 *  encode) failed. A device-side wait that exceeds its time limit makes the
 *  kernel stop early and record RA_ERR_TIMEOUT in the status word, read with
 *  ring_attn_last_error() after synchronising the stream. Nothing throws.
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, N % P != 0, H % G != 0, misaligned,
                               a written range overlapping another argument, or a device
                               pointer that is not memory of the current device */
  RA_ERR_UNSUPPORTED = 2,   /* head_dim not in {64, 128}, no sm_103a device, or a size past a
                               launch limit (e.g. batch x heads x P x query tiles >= 2^31) */
  RA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  RA_ERR_TIMEOUT = 4,       /* a device-side wait ran out (read via ring_attn_last_error) */
  RA_ERR_BOUNDS = 5         /* debug builds only (RA_DEBUG): a kernel's index check failed and
                               the access was skipped (read via ring_attn_last_error) */
} ra_status;

/* Shard layouts ("Part 4: Ring Attention" §4.3.1 for contiguous; "Ring Attention"
 * (aarnphm.xyz): striped ownership alternates, token t -> shard t mod P; "Part 4"
 * §4.8.3 and Transformer Math "Ring Attention" (aicassindra), "Causal masking
 * wastes half the ring", for zigzag). */
typedef enum {
  RA_LAYOUT_CONTIGUOUS = 0, /* shard u = tokens [u*S, (u+1)*S), local i -> token u*S + i */
  RA_LAYOUT_STRIPED = 1,    /* token t -> shard t mod P, local index t div P */
  RA_LAYOUT_ZIGZAG = 2      /* 2P chunks of C = N/(2P): shard u = chunk u (local 0..C-1)
                               then chunk 2P-1-u (local C..2C-1); needs N % (2P) == 0 */
} ra_layout;

/* Element type of the output O (ra_problem.o_dtype). bf16 is the usual attention
 * output. fp32 keeps the fp32 result of the division O = y / z. Rounding O to bf16
 * adds up to half a bf16 unit in the last place: 0.0078 for 2 <= |O| < 4 and
 * 0.0156 for 4 <= |O| < 8, so an absolute error bound of 1e-2 at every magnitude
 * holds only for the fp32 output. Both are results of the same computation (bf16
 * inputs, fp32 accumulation). */
typedef enum { RA_DTYPE_BF16 = 0, RA_DTYPE_F32 = 1 } ra_dtype;

/* Tile classes of a (query tile, key tile) pair ("Part 4" §4.8.1 "Skipping
 * Fully-Masked Blocks"). */
typedef enum { RA_TILE_EMPTY = 0, RA_TILE_PARTIAL = 1, RA_TILE_FULL = 2 } ra_tile_class;

/* Tile edge (rows and keys) used by the tensor-core kernels and by
 * ring_attn_tile_classes. */
#define RA_TILE 128

typedef struct {
  int32_t batch;      /* B >= 1 */
  int32_t seqlen;     /* N >= 1, N % P == 0 (zigzag: N % 2P == 0), N < 2^30 */
  int32_t heads;      /* H >= 1 */
  int32_t kv_heads;   /* G >= 1, H % G == 0 */
  int32_t head_dim;   /* d in {64, 128} */
  int32_t P;          /* number of virtual shards, 1 <= P <= N */
  int32_t causal;     /* 0 or 1 */
  int32_t layout;     /* ra_layout */
  float scale;        /* score scale; 0 means 1/sqrt(d) */
  int32_t o_dtype;    /* ra_dtype of o (0 = bf16, the default of a zeroed struct); read by
                         ring_attn_fwd, ring_attn_fwd_host, ring_attn_finalize,
                         ring_attn_decode(_noalloc) (written o) and ring_attn_bwd (the saved
                         o it reads); the step calls ignore it */
} ra_problem;

/* Full ring forward: every virtual device u folds all P shards in ring order
 * b = (u - s) mod P, s = 0..P-1, and writes O = y / z (bf16, round to nearest
 * even, or fp32 with p->o_dtype = RA_DTYPE_F32) and LSE = m + ln z (fp32). The
 * bf16 output is exactly the fp32 one rounded. Tiles that the causal mask leaves empty are
 * skipped. Source: "Ring Attention" (aarnphm.xyz), recurrence display and
 * O = y/z; "Part 4: Ring Attention" §4.3 and §4.8.1.
 * q, k, v in; o, lse out (device). Errors: see conventions. */
ra_status ring_attn_fwd(const ra_problem* p, const void* q, const void* k, const void* v,
                        void* o, float* lse, void* stream);

/* The full ring forward for inputs that live in HOST memory: q, k, v are read
 * from, o and lse written to, host memory (page-locked memory lets the copies
 * overlap the kernels; pageable memory also works, with the copies serialised).
 * The work goes through the GPU in pieces — one sequence's query heads of one
 * kv group with that kv head — in as many device slots as the workspace holds
 * (at least two): while piece i is computed on `stream`, the inputs of the next
 * pieces travel in as soon as their slot is free (up to slots - 1 pieces ahead),
 * and the outputs of finished pieces travel out (strided copies gather a group's
 * heads). A host tensor in page-locked memory that the device maps at the same
 * address (ring_attn_host_mapped) is moved by the SMs — small copy kernels
 * on high-priority streams the call creates and releases, whose blocks run ahead of
 * the ring kernel's; copy-engine transfers over the host link were seen to stall for
 * tens of milliseconds while the GPU changed clocks under its power cap, SM loads and
 * stores were not. Other host tensors (pageable memory) go through the copy engines:
 * inputs on `copy_stream`, outputs on a stream of the call's own. Only the first
 * piece's inputs and the last one's outputs are not hidden behind compute. Each piece is exactly a ring_attn_fwd
 * call on its heads (the results equal ring_attn_fwd bit for bit). Work enqueued
 * on `stream` before the call happens before any of its copies, and `stream`
 * completes only once the outputs are in host memory, so synchronising `stream`
 * is enough; that holds after an error returned midway too (`stream` still waits
 * for every copy already queued) before the workspace or host buffers are reused.
 * The call returns after enqueuing; it creates and releases its ordering events
 * and its output stream itself. There is no counterpart in the pages: this is an
 * interface choice of this library (host-resident inputs, e.g. in the CPU memory
 * of a Grace host).
 * q, k, v, o, lse: host pointers in the shapes of ring_attn_fwd. workspace:
 * device memory of this device, 16-byte aligned, overwritten, of at least two
 * slots (ring_attn_fwd_host_workspace_bytes gives room for sixteen). copy_stream:
 * the stream of copy-engine input transfers (pageable inputs); it may equal stream
 * (those transfers then do not overlap the kernels). */
ra_status ring_attn_fwd_host(const ra_problem* p, const void* q, const void* k, const void* v,
                             void* o, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream, void* copy_stream);

/* 1 when ring_attn_fwd_host would move the host range [p, p + bytes) with copy
 * kernels: page-locked memory that the current device maps at the same address,
 * 4-byte aligned, with the whole range inside one allocation or registration (its
 * first and last byte checked, then the extent of the allocation that holds p).
 * 0 otherwise — pageable memory, device memory, a range that runs past the end of
 * its allocation, a null pointer, bytes == 0, or a device that is not sm_103 — and
 * such a tensor goes through the copy engines. A pure query: nothing is launched
 * and no memory is touched. No counterpart in the pages. */
int32_t ring_attn_host_mapped(const void* p, size_t bytes);

/* Recommended bytes of device workspace for ring_attn_fwd_host: sixteen slots (or
 * one per piece if batch * kv_heads is smaller), a slot being one piece's q, k, v,
 * o, lse, each rounded up to 256 bytes. A piece holds seqlen tokens of
 * heads/kv_heads query heads and one kv head. Any workspace of at least two slots
 * is accepted; the call uses as many slots as it holds. Pure host code. */
size_t ring_attn_fwd_host_workspace_bytes(const ra_problem* p);

/* One ring step for all virtual devices at once: device u folds shard
 * b = (u - s) mod P into the running state (m, z, y) of its own query rows.
 * first != 0 starts from the empty state (m = -inf, z = 0, y = 0) and ignores
 * the input contents of m, z, y. State layout: m, z [B, H, N] fp32 with m the
 * running max of the scaled scores (natural units, -inf when nothing was
 * seen), y [B, N, H, d] fp32 unnormalised; rows that shard b leaves fully
 * masked are left unchanged. Calling s over any permutation of 0..P-1 gives
 * the same final state up to rounding ("Ring Attention: Distributed Attention
 * Across Devices", "Building block: the online-softmax trick": any order).
 * Source: "Ring Attention" (aarnphm.xyz), recurrence display (one step).
 * 0 <= s < P. m, z, y are read (unless first) and written (device). */
ra_status ring_attn_step(const ra_problem* p, int32_t s, int32_t first,
                         const void* q, const void* k, const void* v,
                         float* m, float* z, float* y, void* stream);

/* Same contract as ring_attn_step, computed by a plain SIMT fp32 kernel
 * (scores, exponentials and P·V in fp32 without tensor cores or bf16 rounding of
 * the probabilities). A cross-check for the tensor-core kernels; slow. */
ra_status ring_attn_step_simt(const ra_problem* p, int32_t s, int32_t first,
                              const void* q, const void* k, const void* v,
                              float* m, float* z, float* y, void* stream);

/* Running state -> result: O = y / z (bf16, or fp32 with p->o_dtype =
 * RA_DTYPE_F32), LSE = m + ln z (fp32); z = 0 gives
 * O = 0, LSE = -inf. Source: "Ring Attention" (aarnphm.xyz), O = y/z; "Part 4"
 * §4.4 FINAL. m, z, y in; o, lse out (device). */
ra_status ring_attn_finalize(const ra_problem* p, const float* m, const float* z,
                             const float* y, void* o, float* lse, void* stream);

/* Merge n normalised partial results of the same query rows over disjoint key
 * sets: LSE = M + ln sum_p exp(LSE_p - M) with M = max_p LSE_p, and
 * O = sum_p exp(LSE_p - LSE) O_p; parts with LSE_p = -inf contribute nothing,
 * all -inf gives O = 0, LSE = -inf. Source: Transformer Math "Ring Attention"
 * (aicassindra), "The ring is a prefill algorithm" (P partial triples combined
 * by one rescale-and-add reduction); "Ring Attention: what the near-infinite
 * context paper actually says", "What the online softmax accumulation actually
 * does across rounds".
 * o_parts [n, B, N, H, d] fp32, lse_parts [n, B, H, N] fp32 in; o [B, N, H, d]
 * bf16, lse [B, H, N] fp32 out (device). 1 <= n_parts <= 1024. */
ra_status ring_attn_merge(int32_t n_parts, int32_t batch, int32_t seqlen, int32_t heads,
                          int32_t head_dim, const float* o_parts, const float* lse_parts,
                          void* o, float* lse, void* stream);

/* Pass-Q decode: n_q query rows per (batch, head), at global positions
 * q_pos0 .. q_pos0 + n_q - 1, attend to a KV cache of N tokens that stays sharded
 * and stationary in P virtual shards (layout as in p). Phase 1: every virtual
 * device u scores all queries against its own shard only and writes a
 * normalised partial (O_u, LSE_u) into the workspace (a shard is cut into key
 * chunks, each one more partial). Phase 2: the partials are combined by the
 * ring_attn_merge kernel. When a row group's partials come from at most 8 CTAs
 * and the grid is one wave or less, those CTAs run as one thread-block cluster
 * and combine the partials through distributed shared memory instead: one launch,
 * and the workspace is not touched. Under the causal mask a query sees key positions
 * <= its own. Source: Transformer Math "Ring Attention" (aicassindra), "The ring
 * is a prefill algorithm" (broadcast the query, partial per shard, one
 * reduction); "Part 4: Ring Attention" (Fofadiya) §4.9.4.4 (pass-Q).
 * q [B, n_q, H, d] bf16, k, v [B, N, G, d] bf16 in; o [B, n_q, H, d] bf16 and
 * lse [B, H, n_q] fp32 out (o fp32 with p->o_dtype = RA_DTYPE_F32). workspace:
 * caller-owned device memory of at least ring_attn_decode_workspace_bytes(p, n_q)
 * bytes, 16-byte aligned, overwritten. 1 <= n_q <= 4096; with causal = 1,
 * q_pos0 + n_q <= N. One or two launches on stream. */
ra_status ring_attn_decode(const ra_problem* p, int32_t n_q, int32_t q_pos0, const void* q,
                           const void* k, const void* v, void* o, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Bytes of workspace ring_attn_decode needs for this problem and n_q (0 if the
 * arguments are invalid). Pure host code. */
size_t ring_attn_decode_workspace_bytes(const ra_problem* p, int32_t n_q);

/* Size of the fixed device scratch ring_attn_decode_noalloc keeps its partials in. */
#define RA_DECODE_SCRATCH_BYTES (16u << 20)

/* Decode for callers that cannot allocate device memory when they decode (a
 * serving loop that must not stall on an allocator, a plugin whose host owns all
 * device memory, a runtime that plans memory up front). Same contract and result
 * as ring_attn_decode, but the partials go to a fixed scratch array of
 * RA_DECODE_SCRATCH_BYTES bytes in the library's static device memory instead of
 * a caller workspace. There is no counterpart in the pages: this is an interface
 * choice of this library.
 * Returns RA_ERR_INVALID_ARG when ring_attn_decode_workspace_bytes(p, n_q) exceeds
 * RA_DECODE_SCRATCH_BYTES.
 * First call on a device: the CUDA runtime loads modules lazily, so the first call
 * on a device (more exactly: in a device context) loads the module that holds the
 * array, which reserves its RA_DECODE_SCRATCH_BYTES on that device until the
 * process exits, and looks up its address (cudaGetSymbolAddress) with the device
 * current. That call can return RA_ERR_CUDA if the device has no room for the
 * array (no CUDA error is left pending); make it before capturing a stream. Later
 * calls in the same context allocate nothing; a new context (after
 * cudaDeviceReset) repeats the first-call step.
 * All calls on a device share the scratch and each call overwrites it: calls
 * whose work may overlap on the GPU (different streams without ordering) race. */
ra_status ring_attn_decode_noalloc(const ra_problem* p, int32_t n_q, int32_t q_pos0,
                                   const void* q, const void* k, const void* v, void* o,
                                   float* lse, void* stream);

/* Backward of the full ring forward: dQ, dK, dV for an upstream gradient dO,
 * from the forward's inputs and its saved output O and LSE. The K/V blocks
 * circulate a second time carrying their accumulating dK/dV, each query shard
 * adds its contribution as a block passes, and the score blocks are recomputed
 * from the saved per-row statistics rather than stored (Transformer Math "Ring
 * Attention" (aicassindra), "The backward pass costs a second ring"). The ring
 * runs in the reverse direction: at backward step s = 0..P-1 virtual device u
 * holds block (u + s) mod P ("Ring Attention: what the near-infinite context
 * paper actually says", "Production tradeoffs no one mentions in the benchmark
 * post"). With S = scale Q K^T (causal mask as in the forward),
 * A = exp(S - LSE) and D = rowsum(dO * O) per query row:
 *     dV = A^T dO,  dS = A * (dO V^T - D),  dQ = scale dS K,  dK = scale dS^T Q;
 * a kv head's dK, dV sum over the query heads that read it. A row with
 * LSE = -inf contributes nothing. Probabilities and dS are rounded to bf16 for
 * the tensor-core products; accumulation is fp32; dq, dk, dv are written as
 * bf16 (round to nearest even), every element overwritten.
 * q, dout [B, N, H, d] bf16, o [B, N, H, d] bf16 (fp32 with p->o_dtype =
 * RA_DTYPE_F32), k, v [B, N, G, d] bf16, lse [B, H, N] fp32 in;
 * dq [B, N, H, d], dk, dv [B, N, G, d] bf16 out (device). workspace:
 * caller-owned device memory of at least ring_attn_bwd_workspace_bytes(p)
 * bytes, 16-byte aligned, overwritten. Three launches on stream. */
ra_status ring_attn_bwd(const ra_problem* p, const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dout, void* dq, void* dk,
                        void* dv, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace ring_attn_bwd needs for this problem (0 if the problem is
 * invalid): 9 KiB per 128-row query tile of every (batch, head) plus 4 KiB. Pure
 * host code. */
size_t ring_attn_bwd_workspace_bytes(const ra_problem* p);

/* Shard ownership on the HOST: owner[t], local[t] for t < N and
 * token_of[u*S + i] (S = N/P) for the given layout. Pure host code; host
 * pointers, each N int32. Source: as for ra_layout. */
ra_status ring_attn_shard_map(int32_t layout, int32_t seqlen, int32_t P,
                              int32_t* owner, int32_t* local, int32_t* token_of);

/* The same three maps computed on the GPU by the index functions the kernels
 * use; device pointers, each N int32. */
ra_status ring_attn_shard_map_device(int32_t layout, int32_t seqlen, int32_t P,
                                     int32_t* owner, int32_t* local, int32_t* token_of,
                                     void* stream);

/* Tile classes of the shard pair (u, b) as the kernels see them: classes
 * [ceil(S/RA_TILE)][ceil(S/RA_TILE)] int8 (ra_tile_class), counting only rows
 * and keys < S. Computed on the GPU by the kernels' own classifier. Source:
 * "Part 4: Ring Attention" §4.8.1. classes: device pointer. */
ra_status ring_attn_tile_classes(const ra_problem* p, int32_t u, int32_t b, int8_t* classes,
                                 void* stream);

/* Element mask of the shard pair (u, b): mask[i][j] = 1 iff local query i of
 * shard u may attend to local key j of shard b, [S][S] uint8, computed on the
 * GPU by the kernels' own per-row visibility rule. mask: device pointer. */
ra_status ring_attn_mask(const ra_problem* p, int32_t u, int32_t b, uint8_t* mask,
                         void* stream);

/* Reads and clears the calling GPU's status word. *device_code receives the
 * ra_status a kernel recorded (RA_OK if none). Synchronises with the device's
 * legacy stream; call after synchronising the stream of interest. */
ra_status ring_attn_last_error(int32_t* device_code);

/* Launches a one-warp kernel that waits, with the library's bounded wait, on a
 * barrier that nothing completes, for at most limit_ns nanoseconds; it then
 * records RA_ERR_TIMEOUT in the status word and returns. Lets a test see the
 * timeout path without a hang. 0 < limit_ns <= 10^9. */
ra_status ring_attn_selftest_timeout(uint64_t limit_ns, void* stream);

/* Test hook for the kernels' abort path. Sets the time limit of every device-side
 * wait of the forward, step, backward and decode kernels launched by later calls
 * in this process (all devices) to limit_ns nanoseconds; 0 restores the default,
 * 2 s. In the debug build (ring_attn_debug_checks() == 1) every wait tests its
 * barrier without blocking and looks at its limit on every poll (a limit under
 * 1000 ns, below the resolution of the GPU's timer, counts polls), so a limit of a
 * few nanoseconds makes every wait that is not already complete run out on an
 * ordinary problem: the kernel that gives up records RA_ERR_TIMEOUT, stops its
 * other roles through a shared flag, lets the copies and products it has in
 * flight finish (those waits keep their own fixed limit), frees its tensor memory
 * and returns, and its outputs are undefined. The release build's waits first
 * block in hardware for a short, system-defined time, so there only waits longer
 * than that run out. Meant for tests only: an application has no reason to call
 * it. Limits above the default give RA_ERR_INVALID_ARG. */
ra_status ring_attn_selftest_wait_limit(uint64_t limit_ns);

/* 1 if this library was built with the kernels' index checks (RA_DEBUG), else 0.
 * In such a debug build every raw global load or store (one that is not a TMA copy)
 * of the ring, step, backward and decode kernels first checks its index range
 * against its buffer; a failed check records RA_ERR_BOUNDS in the status word and
 * skips the access. (The merge, finalize and index-map kernels address memory only
 * through their launch coordinates under explicit guards, and the host-copy kernels
 * of ring_attn_fwd_host only within ranges the host has checked; they carry no
 * checks.)
 * Results are otherwise those of the release build. No counterpart in the pages. */
int32_t ring_attn_debug_checks(void);

/* Launches one thread that checks the index range [4, 5) against a 4-element
 * extent without accessing memory: a debug build records RA_ERR_BOUNDS in the
 * status word, a release build records nothing. Lets a test see the check path
 * fire without a faulty kernel. */
ra_status ring_attn_selftest_bounds(void* stream);

/* Human-readable name of a status code (static string). */
const char* ra_status_str(ra_status s);

/* The cudaError_t behind the most recent RA_ERR_CUDA that a call of this library
 * returned on the calling host thread (0 before any). A tensor map the driver
 * refused to encode reads cudaErrorInvalidValue. Pure host code. */
int32_t ring_attn_last_cuda_error(void);

/* CUDA's name for a cudaError_t value (cudaGetErrorName; a static string). */
const char* ring_attn_cuda_error_name(int32_t code);

/* Library ABI version (major*100 + minor). */
int32_t ring_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_H */
