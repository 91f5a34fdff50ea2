/*
 * gdn.h - C ABI of the GB300 (sm_103a) gated delta rule prefill library.
 *
 * The operation: for every packed sequence n and value head h, run the
 * gated delta rule
 *
 *     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * over the sequence's rows, starting from a gathered initial state, and
 * write every o_t and the final S.
 *
 * Where it comes from: System1-Omni PR #186 ("Purpose and summary" and the
 * review-map row on device operations) runs the model's linear-attention
 * layers as one batched call in which every candidate sequence keeps its own
 * recurrent state and short continuations start from a prefix's state. The
 * recurrence itself is the gated delta rule of "Gated Delta Networks:
 * Improving Mamba2 with Delta Rule" (ICLR 2025), the open-jev-fast README's
 * reference [5]. The kernels evaluate it in the chunked form that README
 * describes for its GDN kernel (Phase 3 item 1): 64-token chunks, with the
 * gate cumulative sum, the K K^T product, the unit-lower-triangular solve,
 * the u/w products, the chunk output and the state update. q and k are
 * L2-normalised inside the kernel; the README puts that normalisation in its
 * input-prep kernel (Phase 2 item 1). Handing a prefix's final state to each
 * continuation (README Phase 2 item 2) is the initial_state + state_index
 * gather.
 *
 * Conventions shared by every entry point
 *  - All tensors are caller-owned, contiguous, row-major device memory. The
 *    library allocates nothing, never synchronises inside gdn_prefill_varlen,
 *    and launches only on the given stream (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream).
 *  - Value head h reads q/k head h / (h_v / h_qk) (contiguous groups).
 *  - L2 normalisation: x / sqrt(sum x^2 + 1e-6), in fp32, for q and k.
 *  - scale == 0 selects d_k^-1/2.
 *  - Errors found on the host are returned before anything is launched and
 *    nothing is written. Inconsistencies only the device can see (cu_seqlens,
 *    state_index) set a status word in the workspace and leave the outputs
 *    unspecified; the kernels never trap. Read it with gdn_get_device_status.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 1

/* Storage types. */
typedef enum { GDN_BF16 = 0, GDN_F32 = 1 } gdn_dtype;

/* Result codes (the value of the device status word uses the same codes). */
typedef enum {
  GDN_OK = 0,
  GDN_ERR_NULL = 1,           /* a required pointer is NULL */
  GDN_ERR_SHAPE = 2,          /* unsupported or inconsistent sizes */
  GDN_ERR_DTYPE = 3,          /* unsupported storage type */
  GDN_ERR_ALIGN = 4,          /* a pointer is not 16-byte aligned */
  GDN_ERR_SEQLENS = 5,        /* device: cu_seqlens[0] != 0, decreasing, cu[N] != total_tokens,
                                 or a length above max_seqlen */
  GDN_ERR_STATE_INDEX = 6,    /* device: state_index outside [-1, num_state_slots) */
  GDN_ERR_ALIAS = 7,          /* an output overlaps an input */
  GDN_ERR_WORKSPACE = 8,      /* workspace NULL, misaligned or smaller than gdn_workspace_bytes */
  GDN_ERR_ARCH = 9,           /* the current device is not sm_103 */
  GDN_ERR_CUDA = 10,          /* a CUDA runtime call failed (launch, query, copy) */
  GDN_ERR_DEVICE_TIMEOUT = 11, /* device: a bounded wait gave up */
  GDN_ERR_PARENT = 12,         /* device: a parent index outside [-1, n) (gdn_prefill_tree) */
  GDN_ERR_VALUE = 13,          /* an argument outside its range (gdn_gated_rmsnorm: eps) */
  GDN_ERR_BOUNDS = 14          /* device, bounds-checked build only (libgdn_checked.so): an index
                                  outside its buffer; the access was skipped */
} gdn_status;

/* Flags. */
#define GDN_FLAG_NO_L2NORM 0x1u /* use q and k as given (tests of closed forms) */
#define GDN_FLAG_SIMT 0x2u      /* run the CUDA-core (SIMT) kernel instead of the tensor-core one */
/* Tests only (fault injection, gdn_prefill_tree): the work list is reversed, so that
 * children come before their parents. A chain of more sequences than the GPU holds
 * units at once then stalls on ready flags that no CTA will set; every bounded wait
 * runs out, the device status becomes GDN_ERR_DEVICE_TIMEOUT and the kernel returns
 * (outputs unspecified). No fault, trap or hang. Ignored by gdn_prefill_varlen. */
#define GDN_FLAG_TEST_CHILD_FIRST 0x4u
/* Run a single long sequence in one chunk-kernel launch even when the segment scan
 * (see gdn_prefill_varlen) would apply. */
#define GDN_FLAG_NO_SEGMENT 0x8u

/*
 * Problem descriptor. Every field is read on the host at call time; the
 * struct is not retained.
 */
typedef struct {
  int32_t num_seqs;        /* N >= 0 (N = 0 writes nothing) */
  int64_t total_tokens;    /* T = cu_seqlens[N]: a host copy, so the call never syncs */
  int32_t max_seqlen;      /* upper bound on any sequence length, or 0 if unknown */
  int32_t h_qk, h_v;       /* h_qk >= 1, h_v a multiple of h_qk */
  int32_t d_k, d_v;        /* each 64 or 128 */
  gdn_dtype qkv_dtype;     /* GDN_BF16 */
  gdn_dtype gate_dtype;    /* g and beta: GDN_BF16 or GDN_F32 */
  gdn_dtype out_dtype;     /* GDN_BF16 or GDN_F32 */
  int32_t num_state_slots; /* rows of initial_state (ignored when it is NULL) */
  float scale;             /* 0 => d_k^-1/2 */
  uint32_t flags;          /* GDN_FLAG_* */
  void* workspace;         /* caller-owned device memory, 256-byte aligned */
  size_t workspace_bytes;  /* >= gdn_workspace_bytes(desc) */
} gdn_desc;

/* GDN_ABI_VERSION of the loaded library. */
int gdn_abi_version(void);

/*
 * Bytes of device workspace gdn_prefill_varlen needs for this descriptor
 * (depends on the descriptor's sizes and flags only; 0 for a NULL desc). The
 * workspace holds the device status word and the work list. Its contents need
 * no initialisation and are rewritten by every call; size it once for the
 * largest batch and reuse it (one call at a time per workspace).
 *
 * A descriptor of one sequence of at least 4096 rows with d_k == d_v (tensor-core
 * kernel, no GDN_FLAG_NO_SEGMENT) also gets room for the segment scan: about
 * 22 fp32 states of h_v x d_k x d_v (44 MiB at h_v = 32, d = 128).
 */
size_t gdn_workspace_bytes(const gdn_desc* desc);

/*
 * Gated delta rule prefill over N packed sequences.
 *
 *  q, k          [T, h_qk, d_k]  bf16
 *  v             [T, h_v,  d_v]  bf16
 *  g             [T, h_v] natural-log decay per token and value head (any finite value)
 *  beta          [T, h_v] write strength (used as given)
 *  cu_seqlens    [N+1] int32, device: sequence n owns rows cu[n] .. cu[n+1]-1
 *  initial_state [num_state_slots, h_v, d_k, d_v] fp32, or NULL (all sequences start from 0)
 *  state_index   [N] int32, device: sequence n starts from initial_state[state_index[n]];
 *                -1 selects a zero state; several sequences may name one slot. NULL means
 *                slot n for sequence n (then num_state_slots >= N, else GDN_ERR_SHAPE).
 *                Ignored when initial_state is NULL.
 *  out           [T, h_v, d_v] out_dtype: o_t for every row
 *  final_state   [N, h_v, d_k, d_v] fp32: S after each sequence's last row (S_0 for an
 *                empty sequence), or NULL to skip
 *
 * Pointers q, k, v, out, initial_state, final_state must be 16-byte aligned;
 * g and beta 4-byte aligned. out must not overlap any input; final_state must
 * not overlap initial_state (one slot can feed many sequences). Asynchronous on
 * `stream`; safe to capture in a CUDA graph (fixed launch shapes for a fixed
 * descriptor, no allocation, no host synchronisation).
 *
 * Segment scan. The chunks of one (sequence, value head) pair form a chain, so a
 * single sequence keeps only h_v SMs busy. When the descriptor qualifies (see
 * gdn_workspace_bytes) and its workspace holds the larger size, a single sequence
 * is cut into segments whose state maps S -> Phi S + Delta (linear in the starting
 * state) are computed side by side and then composed; the segments are then rerun
 * from their true starting states. Results agree with the single-launch path
 * within rounding. A smaller workspace, or GDN_FLAG_NO_SEGMENT, keeps one launch.
 */
gdn_status gdn_prefill_varlen(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const int32_t* cu_seqlens,
                              const float* initial_state, const int32_t* state_index, void* out,
                              float* final_state, const gdn_desc* desc, void* stream);

/*
 * The segment plan gdn_prefill_varlen takes for this descriptor on a device with `sms`
 * SMs: *segments = G, the number of segments (0: one launch), *rows0 = the rows of
 * segment 0, *rows = the rows of each of the G - 1 later segments (rows0 + (G - 1) rows
 * = total_tokens). G > 0 only when the descriptor qualifies (gdn_workspace_bytes) and
 * desc->workspace_bytes holds the larger size. The plan minimises the two launches'
 * makespan in chunk periods (longest-first list scheduling of whole (segment, head)
 * units) and is used only when it beats one launch by more than 15%. Host only, no
 * device call; GDN_ERR_NULL for a NULL argument, GDN_ERR_VALUE for sms < 1.
 */
gdn_status gdn_segment_plan(const gdn_desc* desc, int32_t sms, int32_t* segments, int64_t* rows0,
                            int64_t* rows);

/*
 * Largest num_seqs gdn_prefill_varlen_noalloc accepts. Its built-in scratch
 * (the status word and the work list for this many sequences) takes
 * 256 + 4 * GDN_NOALLOC_MAX_SEQS = 65,792 bytes of static device memory on
 * each device the library is loaded on.
 */
#define GDN_NOALLOC_MAX_SEQS 16384

/*
 * gdn_prefill_varlen without a caller-supplied workspace. The method itself
 * has no counterpart to this call: it is a convenience of this library.
 *
 * Who needs it: callers that cannot hand the library a device buffer, for
 * example
 *  - an operator or plug-in interface that passes only the operation's own
 *    tensors and gives the operator no allocator and no state kept between
 *    calls, so there is nowhere to keep a workspace;
 *  - a serving process that reserves its device memory up front (states,
 *    caches) and owns every later allocation through its own arena;
 *  - code that must not call cudaMalloc or cudaFree on its critical path,
 *    since those calls can synchronise the device and stall other streams.
 *
 * Arguments, layouts, results and host-side errors are those of
 * gdn_prefill_varlen; desc->workspace and desc->workspace_bytes are ignored.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library
 * call): the workspace is a fixed array compiled into the library as static
 * device memory, one per device.
 *
 *  - Set-up: the first call on each device looks up that array's device
 *    address (cudaGetSymbolAddress) and keeps it; GDN_ERR_CUDA if the lookup
 *    fails. Make that first call on a device before any stream capture
 *    starts. The kept address belongs to the device's primary context: after
 *    cudaDeviceReset the call must not be used again in that process.
 *  - Limit: num_seqs > GDN_NOALLOC_MAX_SEQS returns GDN_ERR_WORKSPACE before
 *    anything is launched or written.
 *  - Nothing to clear: every call's first kernel resets the status word and
 *    rewrites the whole work list before the chunk kernel reads them.
 *  - One array per device, shared by every call on it: calls whose work can
 *    overlap on the device (different streams, or host threads whose streams
 *    are not ordered by events) race on it, and their outputs are then
 *    unspecified. Issue such calls on one stream, or order them.
 *  - The device status word of this call lives in that array, and no entry
 *    point reads it back: device-detected errors (GDN_ERR_SEQLENS,
 *    GDN_ERR_STATE_INDEX, GDN_ERR_DEVICE_TIMEOUT) leave the outputs
 *    unspecified without being reported. Callers that need them should use
 *    gdn_prefill_varlen with their own workspace.
 */
gdn_status gdn_prefill_varlen_noalloc(const void* q, const void* k, const void* v,
                                      const void* g, const void* beta,
                                      const int32_t* cu_seqlens, const float* initial_state,
                                      const int32_t* state_index, void* out, float* final_state,
                                      const gdn_desc* desc, void* stream);

/*
 * Bytes of device workspace gdn_prefill_tree needs for this descriptor (0 for a
 * NULL desc): the status word, the work list, a work counter and one ready flag
 * per (sequence, value head). Like gdn_workspace_bytes, it needs no
 * initialisation and is rewritten by every call.
 */
size_t gdn_tree_workspace_bytes(const gdn_desc* desc);

/*
 * A prefix tree of sequences in one launch: sequence n continues from the final
 * state of sequence parent[n], computed by the same call.
 *
 * Where it comes from: System1-Omni PR #186 ("Purpose and summary") runs short
 * continuations from a prefix's state; the open-jev-fast README (Phase 2 item
 * 2, "Prefix tree") hands a long prompt's final recurrent state to each
 * candidate, and its project page draws the two-level tree of the example
 * request (shared context, question branches, candidate tails). With
 * gdn_prefill_varlen such a tree takes one call per level; here the levels run
 * in one launch, and a child's value head starts its state step as soon as its
 * parent's final state for that head is written (its chunk preparation, which
 * does not depend on the state, starts earlier still).
 *
 * Arguments are those of gdn_prefill_varlen plus
 *  parent [N] int32, device: parent[n] in [-1, n). A sequence with parent -1 starts
 *         from initial_state[state_index[n]] (or zero) exactly as in
 *         gdn_prefill_varlen; any other starts from final_state[parent[n]].
 * final_state is required (it carries the states handed from parent to child) and
 * desc->workspace must hold gdn_tree_workspace_bytes(desc) bytes. A parent index
 * outside [-1, n) sets GDN_ERR_PARENT in the device status word (the outputs are
 * then unspecified); a child whose parent never finishes gives up after a bounded
 * wait with GDN_ERR_DEVICE_TIMEOUT. The tensor-core kernel only: GDN_FLAG_SIMT
 * returns GDN_ERR_SHAPE. Asynchronous on `stream`, no allocation, no host
 * synchronisation.
 */
gdn_status gdn_prefill_tree(const void* q, const void* k, const void* v, const void* g,
                            const void* beta, const int32_t* cu_seqlens, const int32_t* parent,
                            const float* initial_state, const int32_t* state_index, void* out,
                            float* final_state, const gdn_desc* desc, void* stream);

/*
 * Synchronises `stream`, then returns the device status word the last call on
 * this workspace left (GDN_OK if the device found nothing), or GDN_ERR_CUDA if
 * the synchronisation or the read failed.
 */
gdn_status gdn_get_device_status(const gdn_desc* desc, void* stream);

/*
 * Gated RMSNorm of the prefill output, one row per token and value head:
 *
 *     y[r, j] = weight[j] * o[r, j] / sqrt(mean_j o[r, j]^2 + eps) * silu(z[r, j]),
 *     silu(z) = z / (1 + exp(-z)),
 *
 * with every step in fp32 and one rounding to y's type (so a row's sum of squares
 * must stay inside fp32: entries up to about 1e18 in magnitude). The open-jev-fast README
 * lists the gated RMSNorm among the six fused element-wise kernels of a layer
 * (Phase 2 item 1) that follow the Gated DeltaNet core, and reports fusing it into
 * that core as measured and rejected (item 4). It gives no formula; this is the
 * textbook RMS normalisation over the d_v entries of a row with a per-channel
 * weight shared by the value heads and a SiLU gate.
 *
 *  o, y    [rows, d_v] (rows = tokens x value heads, e.g. the [T, h_v, d_v] output
 *          of gdn_prefill_varlen), storage type x_dtype (GDN_BF16 or GDN_F32)
 *  z       [rows, d_v] gate, storage type z_dtype (GDN_BF16 or GDN_F32)
 *  weight  [d_v] fp32
 *  d_v     64, 128 or 256; rows >= 0 (0 launches nothing and returns GDN_OK
 *          whatever the pointers); eps > 0 and finite, else GDN_ERR_VALUE
 *
 * Every pointer is caller-owned device memory, 16-byte aligned (GDN_ERR_ALIGN).
 * y may be o itself (in place) but may not overlap o otherwise, nor z or weight
 * (GDN_ERR_ALIAS). Asynchronous on `stream`; no allocation, no workspace.
 */
gdn_status gdn_gated_rmsnorm(const void* o, const void* z, const float* weight, void* y, int64_t rows,
                             int32_t d_v, gdn_dtype x_dtype, gdn_dtype z_dtype, float eps, void* stream);

/* Sizes of a gdn_input_prep call. */
typedef struct {
  int32_t num_seqs;        /* N >= 0 packed sequences */
  int64_t total_tokens;    /* T >= 0 rows; T must equal cu_seqlens[N]; N == 0 needs T == 0 */
  int32_t h_qk, h_v;       /* q/k heads and value heads (>= 1) */
  int32_t d_k, d_v;        /* head sizes, multiples of 8 */
  int32_t conv_width;      /* K, the convolution's taps: 2, 3 or 4 */
  int32_t num_state_slots; /* rows of conv_state_in (0 when it is NULL) */
} gdn_prep_desc;

/*
 * GDN input prep: the steps in front of gdn_prefill_varlen that the open-jev-fast
 * README fuses into one "Gated DeltaNet input prep" kernel (Phase 2 item 1):
 * causal depthwise convolution and SiLU over the packed projection rows, the
 * q / k / v split and the gate parameters. With C = 2 h_qk d_k + h_v d_v
 * channels, for each sequence n (rows [cu[n], cu[n+1])) and channel c:
 *
 *     u[t, c] = silu(conv_bias[c] + sum_{j<K} conv_w[c, j] x[t - (K-1) + j, c])
 *     q = u[:, 0 : h_qk d_k],  k = u[:, h_qk d_k : 2 h_qk d_k],  v = u[:, 2 h_qk d_k :]
 *     g[t, h] = -exp(A_log[h]) ln(1 + exp(a[t, h] + dt_bias[h])),  beta = 1 / (1 + exp(-b))
 *
 * where rows before a sequence's first row read its carried window (so that a
 * continuation sees the prefix's last rows, as the README's prefix tree requires).
 * The README gives neither the channel layout nor the gate formula: channels are
 * taken as contiguous q | k | v blocks, and the gates as the decay of "Gated Delta
 * Networks: Improving Mamba2 with Delta Rule" (the README's reference [5]), which
 * keeps Mamba2's form. Head expansion and the q/k L2 norm stay in the prefill
 * (value head h reads q/k head h / (h_v / h_qk); gdn_prefill_varlen normalises).
 *
 *  x               [T, C] bf16, the packed projection rows
 *  conv_w          [C, K] fp32 (tap K-1 multiplies the current row); conv_bias [C]
 *                  fp32 or NULL
 *  cu_seqlens      [N+1] int32 (device), as in gdn_prefill_varlen; inconsistent
 *                  values give unspecified outputs but no access out of bounds
 *  conv_state_in   [num_state_slots, K-1, C] bf16 or NULL: the K-1 rows that precede
 *                  each sequence, oldest first, slot state_index[n] (NULL: slot n;
 *                  a negative or out-of-range index, or NULL conv_state_in: zeros)
 *  a, b            [T, h_v] bf16, the gate projections, or a = NULL to skip the gates
 *                  (then b, A_log, dt_bias, g and beta are not used)
 *  A_log, dt_bias  [h_v] fp32
 *  q, k            [T, h_qk, d_k] bf16 out; v [T, h_v, d_v] bf16 out
 *  g, beta         [T, h_v] fp32 out (ready for gdn_prefill_varlen with fp32 gates)
 *  conv_state_out  [N, K-1, C] bf16 out or NULL: each sequence's last K-1 input rows
 *                  (reaching into its carried window when it is shorter)
 *
 * Arithmetic in fp32; q, k and v are rounded to bf16 once, after SiLU. x, conv_w,
 * q, k, v and both conv states must be 16-byte aligned, the other fp32 and int32
 * arrays 4-byte aligned (GDN_ERR_ALIGN); no output may overlap an input or another output
 * (GDN_ERR_ALIAS). Asynchronous on `stream` (two launches); no allocation.
 */
gdn_status gdn_input_prep(const void* x, const float* conv_w, const float* conv_bias, const int32_t* cu_seqlens,
                          const void* conv_state_in, const int32_t* state_index, const void* a, const void* b,
                          const float* A_log, const float* dt_bias, void* q, void* k, void* v, float* g,
                          float* beta, void* conv_state_out, const gdn_prep_desc* desc, void* stream);

/*
 * gdn_input_prep over a prefix tree: sequence n continues sequence parent[n]
 * (int32 [N], device, parent[n] in [-1, n), as in gdn_prefill_tree), so the rows
 * before its first row are the last rows of its ancestors' path in x (reaching
 * into the root's carried window when that path is shorter than K-1); roots read
 * their carried window as in gdn_input_prep. The window a continuation sees is
 * then the one the open-jev-fast README's replicated full-path layout gives it
 * (Phase 2 item 2). A parent outside [-1, n) is taken as -1 (gdn_prefill_tree
 * reports it). parent may not overlap an output (GDN_ERR_ALIAS) and must be
 * 4-byte aligned; everything else as in gdn_input_prep.
 */
gdn_status gdn_input_prep_tree(const void* x, const float* conv_w, const float* conv_bias, const int32_t* cu_seqlens,
                               const int32_t* parent, const void* conv_state_in, const int32_t* state_index,
                               const void* a, const void* b, const float* A_log, const float* dt_bias, void* q,
                               void* k, void* v, float* g, float* beta, void* conv_state_out,
                               const gdn_prep_desc* desc, void* stream);

/* A static, human-readable name for a status code. */
const char* gdn_status_string(gdn_status s);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
