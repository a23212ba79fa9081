/*
 * upipe.h - C ABI of a single-GPU (sm_103a) library for exact causal (GQA) self-attention,
 * forward and backward, over very long sequences.
 *
 * The schedule follows two published designs:
 *   - UPipe head chunking: attention heads are processed one group of `head_chunk` q-heads at
 *     a time, every group reusing the same workspace ("Road to 5 million sequence length"
 *     talk, UPipe passage; "Road to 5 Million Tokens" summary, section 2, item 6; UPipe
 *     abstract, arXiv 2602.21196).
 *   - FPDT sequence trunking: a query trunk folds key/value trunks 0..m into running
 *     softmax statistics; key/value trunks may live in pinned host memory and are staged
 *     into two device slots on a side copy stream while the previous trunk computes
 *     ("Training Ultra Long Context LM with Fully Pipelined Distributed Transformer",
 *     Key Findings items 1-3 and Technical Deep Dive).
 *   - DeepSpeed Ulysses' head<->sequence all-to-all becomes, on one GPU, the
 *     `upipe_seq_to_head_major` gather into the group workspace (FPDT talk, Technical Deep
 *     Dive, first paragraph); the inverse scatter is fused into the kernels' epilogues.
 *
 * Definition computed (per batch b, q-head h, kv-head c = h / (Hq/Hkv), scale = 1/sqrt(D)):
 *   s_ij = scale <q_i, k_j>, j <= i when causal;  P = row softmax(s);  O = P V;
 *   LSE_i = ln sum_j exp(s_ij);  and the analytic gradients dQ, dK, dV of <dO, O>.
 *
 * Conventions shared by every entry point
 *   - bf16 tensors are passed as `void*` / `const void*` to bf16 (IEEE bfloat16) data.
 *   - Token-major layouts: q, o, dout, dq are [B, S, Hq, D]; k, v, dk, dv are [B, S, Hkv, D],
 *     all dense row-major. lse is float32 [B, Hq, S], natural log.
 *   - Every pointer must be 16-byte aligned. The device pointers of one call must all belong
 *     to one device; k and v may instead both be PINNED host memory
 *     (cudaHostAlloc / cudaHostRegister), which selects the staged host-K/V path.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). All work is enqueued on it
 *     and calls return before the GPU finishes (asynchronous, like a kernel launch).
 *   - Devices: each call runs on the device its device tensors belong to, and leaves the
 *     caller's current device as it found it. Per-device state (copy streams, status word,
 *     each kernel's shared-memory size attribute) is created on the first call that uses that
 *     device, under one library lock, so one process may drive several GPUs; the usual
 *     deployment is one process per GPU (torchrun).
 *   - Ownership: the caller owns every buffer, including the workspace. Per call the library
 *     allocates no device memory. Per device it lazily creates two internal copy streams for
 *     the attention calls and two for the sequence-tiled calls (used only when activations
 *     are pinned host memory), a few events and a 256-byte device status word;
 *     upipe_shutdown() releases them.
 *   - Errors: all arguments are validated before anything is enqueued; on an argument error
 *     nothing is launched and a status code is returned (see upipe_status). A CUDA call that
 *     fails part-way through a call (UPIPE_ERR_CUDA) returns at once: work already enqueued,
 *     including copies on the library's copy streams, still runs, so synchronise the device
 *     before reusing or freeing that call's buffers; its outputs are undefined. A device-side
 *     bounded wait that expires sets the device status word and the kernel exits early; the
 *     host learns of it through upipe_sync_status(). Asynchronous CUDA faults surface at the
 *     caller's next synchronisation.
 */
#ifndef UPIPE_H_
#define UPIPE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  UPIPE_OK = 0,
  UPIPE_ERR_INVALID_ARG = 1,          /* bad shape, pointer, alignment or placement */
  UPIPE_ERR_UNSUPPORTED = 2,          /* valid request outside what the kernels implement */
  UPIPE_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes < upipe_workspace_bytes(...) */
  UPIPE_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed */
  UPIPE_ERR_TIMEOUT = 5               /* a kernel's bounded wait expired (see sync_status) */
} upipe_status;

/* Which pass a workspace is sized for. UPIPE_PASS_FUSED: the loss's one-call forward and
 * backward (upipe_ce_fwd_bwd); every other workspace query returns 0 for it. */
enum { UPIPE_PASS_FWD = 0, UPIPE_PASS_BWD = 1, UPIPE_PASS_BOTH = 2, UPIPE_PASS_FUSED = 3 };

/* What may live in pinned host memory (bits of upipe_workspace_bytes' host_mask):
 * UPIPE_HOST_KV: k and v (and then dk, dv); UPIPE_HOST_ACT: q and o in the forward, q, o, dout
 * and dq in the backward (each independently of the others). */
enum { UPIPE_HOST_KV = 1, UPIPE_HOST_ACT = 2 };

/*
 * Bytes of device workspace one upipe_attn_fwd / upipe_attn_bwd call needs.
 * Pure host arithmetic; touches no device. Returns 0 for arguments that the matching
 * attention call would reject. Every term is proportional to head_chunk (q-heads) or to
 * head_chunk/(Hq/Hkv) (kv-heads), so the workspace of a chunked call is head_chunk/Hq of the
 * unchunked one at the same seq_trunk - the activation-memory cut UPipe reports (UPipe
 * abstract, arXiv 2602.21196: up to 87.5% for a 32B model, i.e. 8 of 64 heads).
 *   pass: UPIPE_PASS_FWD, UPIPE_PASS_BWD or UPIPE_PASS_BOTH (the max of the two).
 *   host_mask: UPIPE_HOST_KV if k/v will be pinned host memory (two trunk slots instead of
 *     full K/V; the forward then walks key/value trunks outermost, staging each once, and
 *     keeps every query trunk's fp32 running state: head_chunk*S*(D+2)*4 bytes per batch
 *     row; the backward also reserves two dK and two dV trunk slots, used when dk/dv are
 *     pinned host memory as well). | UPIPE_HOST_ACT if any of q, o, dout, dq will be pinned
 *     host memory (per pass, a few head-group-sized staging buffers so that each group's
 *     activations move in and out while the neighbouring group computes). 1 keeps meaning
 *     host k/v, as in earlier versions of this interface.
 */
size_t upipe_workspace_bytes(int B, int64_t S, int Hq, int Hkv, int D, int causal,
                             int head_chunk, int64_t seq_trunk, int pass, int host_mask);

/*
 * Forward: o = softmax(scale q k^T + mask) v, lse = ln(sum exp(...)).
 *   q [B,S,Hq,D] bf16 (device or pinned host); k, v [B,S,Hkv,D] bf16 (device, or both pinned
 *     host); o [B,S,Hq,D] bf16 (device or pinned host, written); lse [B,Hq,S] float32
 *     (device, written), or NULL for a prefill (inference) call that keeps no softmax
 *     statistics: then only o is written, by the same kernels. A host q is copied in one head
 *     group at a time on a library copy stream while the previous group computes, and a
 *     host o is copied out one group at a time while the next group computes ("Training Ultra
 *     Long Context LM with Fully Pipelined Distributed Transformer", Key Findings: host
 *     offload with double buffering); the caller's stream completes after the last copy.
 *   causal: 1 = key j visible to query i iff j <= i; 0 = full attention.
 *   head_chunk: q-heads per group; must divide Hq and be a multiple of Hq/Hkv (a group owns
 *     whole kv-heads). head_chunk = Hq is the unchunked schedule.
 *   seq_trunk: trunk length T in tokens. T >= S means one trunk; otherwise T % 128 == 0.
 *     The last trunk may be shorter (ragged).
 *   workspace: device buffer of >= upipe_workspace_bytes(..., UPIPE_PASS_FWD, host_mask)
 *     bytes for the placement of this call, 256-byte aligned; contents on entry are ignored
 *     and on exit are undefined.
 *   Supported: D in {64, 128}; any S >= 1; B, Hq, Hkv >= 1 (UNSUPPORTED otherwise).
 */
int upipe_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int64_t S, int Hq, int Hkv, int D, int causal, int head_chunk,
                   int64_t seq_trunk, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward: given the forward's o and lse and the upstream gradient dout, writes
 * dq [B,S,Hq,D], dk and dv [B,S,Hkv,D] (bf16; fully overwritten).
 * P is recomputed from lse (no S x S tensor is stored), D_i = <dout_i, o_i> is formed by a
 * pre-kernel, dq accumulates in a float32 workspace buffer and is converted at the end.
 * Same argument rules as upipe_attn_fwd; workspace sized with UPIPE_PASS_BWD.
 *   dk, dv: device memory; or, when k and v are pinned host memory, both may be pinned host
 *     memory too. Then each key/value trunk's dK/dV (final once its launch ends: the backward
 *     walks key/value trunks outermost) is written to a device slot and copied to the host on
 *     the library's copy stream while the next trunk computes, so no S-sized key/value tensor
 *     lives on the device ("Training Ultra Long Context LM with Fully Pipelined Distributed
 *     Transformer", Key Findings: offloading to host memory with double buffering). The
 *     caller's stream completes only after the last copy; mixed placement is INVALID_ARG.
 */
int upipe_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                   const float* lse, const void* dout, void* dq, void* dk, void* dv,
                   int B, int64_t S, int Hq, int Hkv, int D, int causal, int head_chunk,
                   int64_t seq_trunk, void* workspace, size_t workspace_bytes, void* stream);

/*
 * upipe_attn_fwd without a caller-supplied workspace, for callers that cannot allocate device
 * memory (code running under an allocator or memory pool that owns every device byte, real-time
 * code that forbids allocation after start-up, plugins handed only their inputs and outputs).
 * The pages describe no such call; it has no counterpart there.
 *   - The forward's scratch is a file-scope static device array of 32 MiB, created when the
 *     library's device code is loaded on a GPU and held by every GPU that loads it until the
 *     process exits. Problems whose forward workspace (upipe_workspace_bytes, UPIPE_PASS_FWD,
 *     host_mask = 0) exceeds 32 MiB are rejected with UPIPE_ERR_WORKSPACE_TOO_SMALL; e.g. the
 *     Llama3-8B-shaped layer fits up to S = 8192 with head_chunk = 8.
 *   - No call allocates or frees anything (no cudaMalloc/cudaFree, no allocating library call).
 *   - The first call on a device does the per-device set-up (looks up the array's device
 *     address and clears its status word, a synchronous step); make that first call before any
 *     stream capture.
 *   - Every call shares the one array, which keeps the last call's contents. Calls whose GPU
 *     work overlaps (different streams, or unordered host threads) race on it: serialise them.
 *   - Arguments as upipe_attn_fwd with two restrictions and no workspace: q, k, v, o and lse
 *     must all be non-null device memory of one device (no pinned-host staging, and no
 *     prefill form with lse = NULL), else UPIPE_ERR_INVALID_ARG. Shape errors return the same
 *     status as upipe_attn_fwd (UPIPE_ERR_INVALID_ARG or UPIPE_ERR_UNSUPPORTED), checked
 *     before any device access. The result is bitwise the one upipe_attn_fwd gives for the
 *     same arguments with device-resident tensors (same kernels, same arena layout).
 *   - check_status != 0 first synchronises `stream` and returns UPIPE_ERR_TIMEOUT if a kernel
 *     of an earlier call of this function gave up on a bounded wait (blocking; pass 0 to
 *     enqueue without waiting).
 *   - The caller's current device is left as it was.
 */
int upipe_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int64_t S, int Hq, int Hkv, int D, int causal, int head_chunk,
                           int64_t seq_trunk, int check_status, void* stream);

/*
 * Layout transforms standing in for the Ulysses all-to-all on one GPU (HBM-bound copies).
 *   seq_to_head_major: src token-major [B,S,H,D] -> dst head-major [B,h_count,S,D] holding
 *     heads [h_begin, h_begin+h_count).
 *   head_to_seq_major: the inverse; writes only those heads of dst [B,S,H,D].
 * bf16, device pointers, 16-byte aligned; D must be a multiple of 8.
 */
int upipe_seq_to_head_major(const void* src, void* dst, int B, int64_t S, int H, int D,
                            int h_begin, int h_count, void* stream);
int upipe_head_to_seq_major(const void* src, void* dst, int B, int64_t S, int H, int D,
                            int h_begin, int h_count, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status word.
 * Returns UPIPE_OK, UPIPE_ERR_TIMEOUT (a kernel's bounded wait expired since the last
 * check) or UPIPE_ERR_CUDA (the synchronisation itself failed).
 */
int upipe_sync_status(void* stream);

/* Static, human-readable name of a status code. */
const char* upipe_status_string(int status);

/* Detail of the last error on the calling thread ("" if none). Valid until the next call. */
const char* upipe_last_error_message(void);

/* Releases the per-device copy streams, events and status words. Optional at exit. */
void upipe_shutdown(void);

/* ---- Sequence tiling: language-model readout + cross-entropy loss ----------------------
 *
 * The per-token loss is computed seq_tile tokens at a time, so that no buffer has the whole
 * sequence along one dimension ("Road to 5 million sequence length" talk notes, Arctic
 * sequence-tiling passage: element-wise computations such as the loss are chunked along the
 * sequence; "Road to 5 Million Tokens" summary, section 2 item 5, "Sequence Tiling").
 * Definition, for tokens i < S and vocabulary rows j < V:
 *   logits[i][j] = <h_i, w_j>;   lse[i] = ln sum_j exp(logits[i][j]);
 *   loss[i] = lse[i] - logits[i][target[i]], and 0 when target[i] < 0 (an ignored token);
 *   backward, for g[i] = d(total)/d(loss[i]) (the caller's reduction, e.g. 1/count for a mean):
 *   dlogits[i][j] = g[i] (exp(logits[i][j] - lse[i]) - [j == target[i]]) (0 for ignored rows);
 *   dh = dlogits w;   dw = dlogits^T h.
 * The forward stores no logits: each 256-column vocabulary tile leaves a (max, sum) pair per
 * token, merged afterwards. The backward recomputes the logits of one tile of tokens, keeps
 * that tile's dlogits (bf16, seq_tile x V) in the workspace and consumes it in two GEMMs.
 * All GEMMs run on the tensor cores (bf16 operands, fp32 accumulation).
 *
 * Layouts (dense row-major): h [S][Dm] bf16, w [V][Dm] bf16, target [S] int64, loss, lse and
 * dloss [S] float32, dh [S][Dm] bf16, dw [V][Dm] float32 (overwritten with the sum over all
 * tokens). Every pointer: device memory of one device, 16-byte aligned. UPIPE_ERR_UNSUPPORTED
 * unless Dm % 64 == 0, V % 64 == 0, V < 2^31 and seq_tile % 128 == 0; S >= 1 (the last tile
 * may be ragged). A target >= V makes that token's loss (and, in the backward, every
 * gradient) NaN. Workspace: upipe_ce_workspace_bytes (pass as for attention; 0 for a shape
 * the calls reject): forward ceil(V/256) * T' * 8 + T' * 4 bytes with T' = min(seq_tile, S)
 * rounded up to 128; backward min(seq_tile, S) * V * 2 bytes; each rounded up to 256.
 * Asynchronous on `stream`, like the attention calls.
 * Host activations: h (and dh) may instead be PINNED host memory. The call then stages each
 * tile of h into one of two device slots on a library inbound copy stream, two tiles ahead,
 * and copies each tile of dh out on an outbound copy stream while the next tile computes;
 * `stream` completes after the last copy. The workspace must then be sized with host_mask =
 * UPIPE_HOST_ACT, which adds 2 (forward) or 4 (backward) slots of min(seq_tile, S) * Dm * 2
 * bytes, each rounded up to 256 (host_mask 0: device activations only; other bits: 0 bytes).
 * Calls that stage host activations share one pair of copy streams and their events per
 * device: two such calls whose work could overlap (different streams, unordered threads) must
 * be serialised by the caller. Calls with device activations only have no such restriction
 * beyond their workspaces being distinct.
 */
size_t upipe_ce_workspace_bytes(int64_t S, int Dm, int64_t V, int64_t seq_tile, int pass,
                                int host_mask);
int upipe_ce_fwd(const void* h, const void* w, const int64_t* target, float* loss, float* lse,
                 int64_t S, int Dm, int64_t V, int64_t seq_tile, void* workspace,
                 size_t workspace_bytes, void* stream);
int upipe_ce_bwd(const void* h, const void* w, const int64_t* target, const float* lse,
                 const float* dloss, void* dh, float* dw, int64_t S, int Dm, int64_t V,
                 int64_t seq_tile, void* workspace, size_t workspace_bytes, void* stream);
/* Forward and backward in one call, for an upstream gradient dloss known up front (the loss
 * is the last operation: dloss = 1/count for a mean). Per tile the logits GEMM also keeps its
 * fp32 logits (seq_tile x V x 4 bytes of workspace) and one HBM-bound pass turns them into
 * dlogits after the merge, so the backward's logits recompute - a quarter of the two calls'
 * tensor work - is not done. loss, lse, dh and dw are bitwise those of upipe_ce_fwd followed
 * by upipe_ce_bwd. Workspace: upipe_ce_workspace_bytes(..., UPIPE_PASS_FUSED, host_mask) =
 * the forward's partials + T*V*4 (logits) + T*V*2 (dlogits) bytes, T = min(seq_tile, S),
 * each rounded up to 256, plus 4 staging slots with UPIPE_HOST_ACT (h in, dh out). */
int upipe_ce_fwd_bwd(const void* h, const void* w, const int64_t* target, const float* dloss,
                     float* loss, float* lse, void* dh, float* dw, int64_t S, int Dm, int64_t V,
                     int64_t seq_tile, void* workspace, size_t workspace_bytes, void* stream);

/* ---- Sequence tiling: gated (SwiGLU) MLP ------------------------------------------------
 *
 * The MLP is the other per-token computation the same passages chunk along the sequence.
 * Computed seq_tile tokens at a time, so the [S][F] intermediates never exist; each tile's
 * intermediates are recomputed in the backward rather than kept. Definition (no biases;
 * silu(z) = z / (1 + e^-z)):
 *   g = x Wg^T, u = x Wu^T, a = silu(g) * u, y = a Wd^T;
 *   backward, for dy: da = dy Wd, dg = da * u * silu'(g), du = da * silu(g),
 *   dx = dg Wg + du Wu, dWd = dy^T a, dWg = dg^T x, dWu = du^T x.
 * Layouts (dense row-major, bf16 unless noted): x, y, dy, dx [S][Dm]; w_gu [2F][Dm] = Wg
 * (rows 0..F-1) stacked on Wu (rows F..2F-1); w_d [Dm][F]; dw_gu float32 [2F][Dm] and dw_d
 * float32 [Dm][F], both overwritten with the sum over all tokens. Every pointer: device
 * memory of one device, 16-byte aligned. UPIPE_ERR_UNSUPPORTED unless Dm % 64 == 0,
 * F % 128 == 0 and seq_tile % 128 == 0; S >= 1 (ragged last tile). All six GEMMs of a tile
 * run on the tensor cores (bf16 operands, fp32 accumulation); a, g, u, dg, du are rounded to
 * bf16 between GEMMs. Workspace (upipe_mlp_workspace_bytes): forward T*F*2 bytes (a),
 * backward 5*T*F*2 (a, g|u, dg|du), T = min(seq_tile, S), each buffer rounded up to 256;
 * pass BOTH is the larger of the two.
 * Host activations: x, y, dy and dx may each instead be PINNED host memory, staged tile by
 * tile as for the loss (inputs two tiles ahead on an inbound copy stream, outputs copied out
 * while the next tile computes). host_mask = UPIPE_HOST_ACT then adds two slots of
 * T * Dm * 2 bytes for each of x and y (forward) or x, dy and dx (backward).
 */
size_t upipe_mlp_workspace_bytes(int64_t S, int Dm, int F, int64_t seq_tile, int pass,
                                 int host_mask);
int upipe_mlp_fwd(const void* x, const void* w_gu, const void* w_d, void* y, int64_t S, int Dm,
                  int F, int64_t seq_tile, void* workspace, size_t workspace_bytes,
                  void* stream);
int upipe_mlp_bwd(const void* x, const void* w_gu, const void* w_d, const void* dy, void* dx,
                  float* dw_gu, float* dw_d, int64_t S, int Dm, int F, int64_t seq_tile,
                  void* workspace, size_t workspace_bytes, void* stream);

/* ---- Diagnostics ---------------------------------------------------------------------- */

/* Kernel classes for launch counting and profiling. */
enum {
  UPIPE_K_LAYOUT = 0,     /* seq_to_head_major / head_to_seq_major gathers */
  UPIPE_K_ATTN_FWD = 1,   /* forward attention kernel */
  UPIPE_K_BWD_PRE = 2,    /* D = rowsum(dO * O) + dO gather + LSE prescale */
  UPIPE_K_ATTN_BWD = 3,   /* backward attention kernel */
  UPIPE_K_DQ_CONVERT = 4, /* dq float32 -> bf16 token-major */
  UPIPE_K_OTHER = 5,      /* self-tests */
  UPIPE_K_LOSS_GEMM = 6,  /* sequence-tiled loss and MLP: tensor-core GEMMs + epilogues */
  UPIPE_K_LOSS_MERGE = 7, /* sequence-tiled loss: per-token merge, stored logits -> dlogits */
  UPIPE_K_KV_H2D = 8,     /* not a kernel: one key/value trunk staged host -> device (copy
                             stream; "launches" counts trunks) */
  UPIPE_K_DKDV_D2H = 9,   /* not a kernel: one trunk's dK/dV copied device -> host */
  UPIPE_K_KV_WAIT = 10,   /* not a kernel: how long the compute stream stalled waiting for a
                             staged key/value trunk (the copy time not hidden behind compute) */
  UPIPE_K_COUNT = 11
};

typedef struct {
  double total_ms;   /* summed CUDA-event time of the recorded launches */
  uint64_t launches; /* launches recorded */
} upipe_kernel_stat;

/*
 * Test hook for failure handling: n >= 1 arms the n-th host<->device staging copy issued from
 * now on (K/V trunks, dK/dV trunks, head-group activations, tiles of the sequence-tiled
 * calls; counted across calls and threads) to fail as if its copy call had returned an error:
 * the call that would issue it returns UPIPE_ERR_CUDA ("injected staging copy failure")
 * without issuing it. Work that call already enqueued stays enqueued and completes; its
 * outputs are undefined. Fires once, then disarms; 0 disarms; n < 0 is UPIPE_ERR_INVALID_ARG.
 * Touches no device.
 */
int upipe_debug_fail_copy_after(int n);

/* Total kernel launches made by this library in this process (all classes). */
uint64_t upipe_launch_count(void);

/*
 * Profiling: while enabled, every launch is bracketed by CUDA events recorded on the stream
 * it is launched on, and so is each key/value trunk staged in (UPIPE_K_KV_H2D) and each
 * trunk's dK/dV copied out (UPIPE_K_DKDV_D2H) on the library's copy stream, and the compute
 * stream's wait for each staged trunk (UPIPE_K_KV_WAIT).
 * upipe_profile_read() synchronises those events, adds their elapsed times into out[0..n)
 * (indexed by class) and forgets them. Returns a status code. Copies are not counted by
 * upipe_launch_count().
 */
int upipe_profile_enable(int on);
int upipe_profile_read(upipe_kernel_stat* out, int n);

/*
 * Self-test of the tensor-core tile path: one 128 x N x K bf16 MMA tile (fp32 accumulate)
 * computed with the same TMA loads, shared-memory descriptors and TMEM read-back the
 * attention kernels use. c[m][n] = sum_k A(m,k) B(n,k) with
 *   a_mn_major = 0: a is [128][K] row-major;  1: a is [K][128] row-major;
 *   b_mn_major = 0: b is [N][K] row-major;    1: b is [K][N] row-major;
 *   a_manual = 1 stores A into shared memory with the kernels' own swizzled stores instead
 *     of TMA; a_manual = 2 stores A into tensor memory (row m in lane m, two bf16 per
 *     column) and issues the MMA with A read from there (a_mn_major must be 0 for both).
 * N, K in {64, 128}. lbo/sbo: byte offsets written into the MN-major descriptors.
 * c is float32 [128][N]. Device pointers. Test use only.
 */
int upipe_selftest_umma(const void* a, const void* b, float* c, int N, int K,
                        int a_mn_major, int b_mn_major, int a_manual, int lbo, int sbo,
                        void* stream);

/*
 * Self-test of the bounded device wait: launches one CTA that waits on a shared-memory
 * barrier that nothing completes, with a limit of `limit_us` microseconds (1..2000000).
 * The kernel gives up, sets the status word and returns; a following
 * upipe_sync_status(stream) must report UPIPE_ERR_TIMEOUT.
 */
int upipe_selftest_wait_timeout(int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* UPIPE_H_ */
