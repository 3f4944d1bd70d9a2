/*
 * gla.h — C ABI of the GB300 (sm_103a) forward pass of chunkwise gated linear
 * attention.
 *
 * The operation ("Gated Linear Attention Transformers with Hardware-Efficient
 * Training", §4.1 Eq. 3, computed in the chunkwise form of §4.2-4.3):
 *
 *     S_t = Diag(alpha_t) S_{t-1} + k_t^T v_t,     o_t = q_t S_t,
 *
 * for t = 1..T, independently for every batch row b and head h, starting from
 * S_0 (zero, or a state carried from a previous segment, §2.2). The pass
 * returns O = [o_1 .. o_T] and the final state S_T.
 *
 * Gate modes (all given in log space, log alpha <= 0):
 *   GLA_GATE_NONE        alpha_t = 1: causal linear attention (§2.1 Eq. 1);
 *                        log_g must be NULL.
 *   GLA_GATE_HEAD_SCALAR alpha_t = lambda_h for every t and key: the fixed
 *                        decay of "Lightning Attention-2" (§3.2.1, Alg. 1) and
 *                        RetNet; log_g is float[H] = log(lambda_h).
 *   GLA_GATE_PER_KEY     alpha_t in (0,1]^dk, data dependent (GLA, §4.1);
 *                        log_g is float[B,H,T,dk] = log(alpha_t).
 *   GLA_GATE_TOKEN_SCALAR alpha_t = gamma_t for every key, data dependent:
 *                        G_t = gamma_t 1^T 1, the Mamba-2 / mLSTM / Gated
 *                        Retention rows of the GLA paper's Table 1 (§4.1);
 *                        log_g is float[B,H,T] = log(gamma_t).
 *   GLA_GATE_BILINEAR    G_t = alpha_t^T beta_t (Table 1's DFW row): the
 *                        state update is S_t = G_t (.) S_{t-1} + k_t^T v_t;
 *                        log_g is float[B,H,T,dk] = log(alpha_t) and log_b is
 *                        float[B,H,T,dv] = log(beta_t). CUDA-core path only.
 *
 * Layouts. Every tensor is dense, row-major, last dimension contiguous:
 *   q, k   [B,H,T,dk]   dtype (bf16 or fp32)
 *   v, O   [B,H,T,dv]   dtype
 *   log_g  see above    fp32
 *   S0, ST [B,H,dk,dv]  fp32
 *
 * Ownership. All tensor pointers are device pointers owned by the caller,
 * except in gla_fwd_host(), which takes host pointers. The library keeps none
 * of them after a call returns. It allocates nothing on its own except in
 * gla_fwd(), which takes its workspace from the stream-ordered allocator
 * (cudaMallocAsync / cudaFreeAsync on the given stream), and gla_fwd_host(),
 * which stages through a pool of its own.
 *
 * Asynchrony. Every call but gla_fwd_host() only enqueues work on `stream`
 * and returns; none of them synchronises the device. Argument errors are
 * detected on the host before anything is launched. A kernel whose bounded wait runs out records that in
 * a device-side status word (see gla_device_status) and returns early.
 *
 * Thread safety. Calls may be made concurrently from several host threads.
 * The process-wide state is a per-device cache of the TMA encode entry point
 * and device attributes, and gla_fwd_host()'s streams and memory pool.
 */
#ifndef GLA_H_
#define GLA_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GLA_OK = 0,
    GLA_ERR_INVALID_ARG = 1,  /* null/overlapping/misaligned pointer, bad size, gate/log_g mismatch */
    GLA_ERR_UNSUPPORTED = 2,  /* valid request this build does not handle (chunk size, dk > 768, device) */
    GLA_ERR_CUDA = 3,         /* a CUDA runtime call or a launch failed */
    GLA_ERR_WORKSPACE = 4,    /* workspace missing, too small or could not be allocated */
    GLA_ERR_TIMEOUT = 5       /* a kernel's bounded wait ran out (reported by gla_device_status) */
} gla_status;

typedef enum { GLA_BF16 = 0, GLA_FP32 = 1 } gla_dtype;

typedef enum {
    GLA_GATE_NONE = 0,
    GLA_GATE_HEAD_SCALAR = 1,
    GLA_GATE_PER_KEY = 2,
    GLA_GATE_TOKEN_SCALAR = 3,
    GLA_GATE_BILINEAR = 4
} gla_gate;

/* Which kernels run. AUTO picks the tcgen05 tensor-core path for bf16 inputs
 * with dk in {64,128,256} and dv a multiple of 128 (also dk = 512, as two
 * chunk passes over key halves, for every gate but the bilinear one), and the
 * fp32 CUDA-core path otherwise (always for fp32 inputs). All compute the
 * same function. The forward pass takes any dk and dv that are multiples of
 * 16 with dk <= 768.
 *   GLA_PATH_TENSOR  the tensor-core path, as AUTO plans it (a gate-prep kernel
 *                    writing Q (.) Lambda, K (.) Gamma, the chunk decays and the
 *                    masked intra-chunk scores to the workspace, then the
 *                    chunk-serial pass; a sequence split when B*H is small).
 *                    With dk <= 128 and no gate or a per-head decay the chunk
 *                    pass forms the intra-chunk scores itself: no gate then
 *                    runs no prep kernel and, without a split, needs no
 *                    workspace (gla_fwd_workspace_size returns 0)
 *   GLA_PATH_STAGED  the same, under its explicit name
 *   GLA_PATH_FUSED   per-key gate, bf16, dk = 256, dv in {256, 512}, one pass
 *                    over the sequence: one kernel in which a thread-block
 *                    cluster of the head's dv-tile CTAs prepares the gates and
 *                    scores itself and shares them through distributed shared
 *                    memory; it needs no workspace (gla_fwd_workspace_size
 *                    returns 0), at the cost of speed on this hardware (the
 *                    cross-CTA exchange of every chunk sits on the chain).
 *                    GLA_ERR_UNSUPPORTED for other shapes or gates.
 *   GLA_PATH_SPLIT   backward only (gla_bwd): the 16-row form with split bf16
 *                    operands; GLA_ERR_INVALID_ARG for the forward pass.
 * For the backward, TENSOR names its 64-row chunk form (see gla_bwd). */
typedef enum {
    GLA_PATH_AUTO = 0,
    GLA_PATH_TENSOR = 1,
    GLA_PATH_SIMT = 2,
    GLA_PATH_STAGED = 3,
    GLA_PATH_FUSED = 4,
    GLA_PATH_SPLIT = 5
} gla_path;

typedef struct {
    const void* q;          /* [B,H,T,dk] */
    const void* k;          /* [B,H,T,dk] */
    const void* v;          /* [B,H,T,dv] */
    const float* log_g;     /* see gate modes; NULL iff gate == GLA_GATE_NONE */
    const float* S0;        /* [B,H,dk,dv] or NULL (zero initial state) */
    void* O;                /* [B,H,T,dv], written */
    float* ST;              /* [B,H,dk,dv] or NULL (final state not written); may equal S0 */
    int B, H, T, dk, dv;
    int chunk;              /* primary chunk length: 0 or 64 (64 is used either way) */
    gla_dtype dtype;        /* dtype of q, k, v and O */
    gla_gate gate;
    void* workspace;        /* device scratch of >= gla_fwd_workspace_size() bytes, 256-B aligned */
    size_t workspace_bytes;
    int force_segments;     /* 0: the planner chooses the sequence split; n >= 1: use n segments */
    int path;               /* gla_path */
    const float* log_b;     /* [B,H,T,dv] log(beta_t) for GLA_GATE_BILINEAR, else NULL */
    int window_chunks;      /* 0 (default): exact. n > 0: the sliding-window split, see below */
} gla_fwd_params;

/*
 * The sliding-window split (window_chunks = n > 0; off by default, and not
 * exact). With a gate that decays, a state's influence on later tokens fades
 * by the product of the gates in between, so a state started from zero a long
 * enough window earlier is close to the true one (the FlashQLA talk, the
 * "sliding window" property). When the plan splits the sequence into
 * segments (GLA_PATH_TENSOR / STAGED / AUTO, force_segments or the planner),
 * each segment after the first starts from the state that the n chunks of 64
 * tokens before it leave from a zero start, instead of the exact state that
 * the serial scan over all earlier segments gives; everything older is
 * dropped, the sequence's S0 included once the window lies past it. The
 * first segment starts from S0; S_T is the last segment's end state. The
 * dropped part of segment s's start state is Diag(Gamma_w) S_w, with S_w the
 * exact state at the window's first token and Gamma_w the product of the
 * gates over the window, so the start state's error is at most
 * max_k Gamma_w[k] * |S_w| and vanishes as the window grows. Ignored (the pass
 * stays exact) when the plan has a single segment; the bilinear gate never
 * splits. Negative: GLA_ERR_INVALID_ARG.
 */

/*
 * gla_fwd — the whole forward pass, with the bf16 data type.
 * gate = GLA_GATE_PER_KEY if log_g != NULL, else GLA_GATE_NONE.
 * chunk must be 0 or 64. The workspace comes from cudaMallocAsync on `stream`
 * and is released with cudaFreeAsync on the same stream.
 * Returns GLA_OK once everything is enqueued.
 */
gla_status gla_fwd(const void* q, const void* k, const void* v, const float* log_g,
                   const float* S0, void* O, float* ST,
                   int B, int H, int T, int dk, int dv, int chunk, cudaStream_t stream);

/* gla_fwd_ex — the forward pass described by *p, all stages in order on
 * `stream`. If the plan needs workspace, p->workspace must hold
 * gla_fwd_workspace_size(p) bytes (else GLA_ERR_WORKSPACE). */
gla_status gla_fwd_ex(const gla_fwd_params* p, cudaStream_t stream);

/* Bytes of workspace the plan for *p needs (0 if none). Returns 0 for
 * invalid parameters as well; gla_fwd_ex then reports the error. */
size_t gla_fwd_workspace_size(const gla_fwd_params* p);

/* The plan for *p as separate stages, so that a caller can put events
 * between them: gla_fwd_ex(p) == gla_fwd_stage(p, 0) ... gla_fwd_stage(p, n-1).
 * gla_fwd_num_stages returns n (>= 1), or -1 for invalid parameters.
 * gla_fwd_stage_name returns a static string naming the kernel of stage i. */
int gla_fwd_num_stages(const gla_fwd_params* p);
gla_status gla_fwd_stage(const gla_fwd_params* p, int stage, cudaStream_t stream);
const char* gla_fwd_stage_name(const gla_fwd_params* p, int stage);

/*
 * gla_fwd_noalloc — gla_fwd for callers that cannot allocate device memory.
 * (No counterpart in the papers: this is a deployment convenience.)
 *
 * Some hosts cannot call cudaMalloc/cudaMallocAsync: a framework that has
 * given nearly all device memory to its own pool, a latency-critical loop
 * where allocation is banned because it can synchronise the device, or a
 * plugin interface that offers the kernel no allocator. This entry point
 * takes the same arguments as gla_fwd and allocates nothing; its workspace
 * is a fixed array of GLA_NOALLOC_SCRATCH_BYTES inside the library, which
 * every GPU that loads the library holds until the process exits. The plan
 * never splits the sequence here.
 *
 * Returns GLA_ERR_WORKSPACE, before launching anything, when the call would
 * need more than GLA_NOALLOC_SCRATCH_BYTES of workspace (with a per-key gate
 * and dk = 256 that is about B*H*T > 28,000 token-heads); use gla_fwd_ex with
 * a caller-owned workspace for larger calls. The first call on a device looks
 * up the array's device address (with that device current); make it before
 * any stream capture. All calls on a device share the array: calls that
 * overlap on the GPU race on it, so the caller must order them (one stream,
 * or events between streams).
 */
#define GLA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
gla_status gla_fwd_noalloc(const void* q, const void* k, const void* v, const float* log_g,
                           const float* S0, void* O, float* ST,
                           int B, int H, int T, int dk, int dv, int chunk, cudaStream_t stream);

/*
 * gla_fwd_host — the forward pass described by *p with every tensor pointer
 * (q, k, v, log_g, S0, O, ST) in HOST memory. (No counterpart in the papers:
 * this is a deployment convenience.)
 *
 * The call copies the inputs to the device, runs the pass and copies O and
 * S_T back, one slice of the batch at a time (whole batch rows, or groups of
 * heads of one row when B is small) of about `slice_bytes` of copy traffic
 * each (0: 48 MiB; the last slices are cut smaller), so that the copy-in of
 * one slice, the compute of the one before and the copy-out of the one
 * before that overlap. Host memory may be pinned (page-locked, which the
 * overlap needs) or pageable, with no alignment rule. p->workspace and
 * p->workspace_bytes are ignored.
 *
 * Device memory: three slices' buffers and one workspace, from a memory pool
 * private to the library that keeps its pages between calls so that repeated
 * calls map no memory; gla_host_release() gives them back. The work runs on
 * three streams of the library, after all work already enqueued on `stream`,
 * and `stream` waits for it. Unlike the other entry points the call is
 * synchronous: it returns once O and S_T are written in host memory (or on
 * an error, after the library's streams are idle). Calls on one device take
 * turns. The argument rules are gla_fwd_ex's except pointer alignment.
 */
gla_status gla_fwd_host(const gla_fwd_params* p, size_t slice_bytes, cudaStream_t stream);

/* Returns the pages of the current device's gla_fwd_host pool to the driver. */
gla_status gla_host_release(void);

/*
 * Sequence exchange: one long sequence cut into P consecutive segments, e.g.
 * one per GPU, each device holding its segment's q, k, v and gate.
 *
 * A segment started from a state S_in leaves S_out = Diag(Gamma) S_in + S*,
 * with Gamma the product of alpha_t over the segment's tokens (per key) and S*
 * the state the segment leaves from a zero start: the state S_[0] carried from
 * one segment to the next ("Gated Linear Attention Transformers with
 * Hardware-Efficient Training", §2.2), and the FlashQLA talk's correction of a
 * wrongly started segment by one matrix per rank followed by a short serial
 * recurrence over ranks ("core technical principles"). So each device:
 *   1. gla_segment_pair: its segment's pair (log Gamma, S*), from a zero start;
 *   2. exchanges pairs with the devices before it (the caller's collective:
 *      an all-gather, or a send/recv chain of gla_pair_combine results);
 *   3. gla_pair_scan: S_in = the state entering its segment, from the pairs
 *      of the segments before it and the sequence's initial state S0;
 *   4. gla_fwd_ex with S0 = S_in: its part of O, and (last segment) S_T.
 * Pairs compose as (Gamma_2, S*_2) o (Gamma_1, S*_1) =
 * (Gamma_2 Gamma_1, Diag(Gamma_2) S*_1 + S*_2), an associative operation, so a
 * tree of gla_pair_combine calls gives the same states as the serial scan (up
 * to fp32 rounding). Gamma travels as log Gamma (float[B,H,dk]; for the scalar
 * gates every key holds the same value), so a long segment's decay does not
 * underflow in transit. Each pair is B*H*dk*(dv+1)*4 bytes.
 *
 * gla_segment_pair — the pair of the segment that *p describes (its T tokens;
 * B, H, dk, dv, dtype, gate, log_g, k and v as for gla_fwd_ex). q may be NULL
 * (the pair does not depend on it; when given it must be valid, as the gate
 * prep shared with the forward pass reads it); S0, O and ST are ignored.
 * log_Gamma: device float[B,H,dk], written with the sum over the segment of
 * log alpha_t (T log lambda_h for the per-head gate, 0 without a gate).
 * S_star: device float[B,H,dk,dv], written with the state from a zero start.
 * For bf16 with dk in {64,128,256} (p->path != GLA_PATH_SIMT) the pair comes
 * from the tensor-core gate prep and state-only pass; otherwise from the
 * CUDA-core forward pass, whose O goes to the workspace. p->workspace must
 * hold gla_segment_pair_workspace_size(p) bytes (256-byte aligned), else
 * GLA_ERR_WORKSPACE. T = 0 gives (0, 0). GLA_ERR_UNSUPPORTED for the bilinear
 * gate (its decay is a dk x dv matrix, not a key vector). Outputs may not
 * overlap the inputs or each other. Asynchronous on `stream`.
 */
size_t gla_segment_pair_workspace_size(const gla_fwd_params* p);
gla_status gla_segment_pair(const gla_fwd_params* p, float* log_Gamma, float* S_star, cudaStream_t stream);

/*
 * gla_pair_scan — the states entering P consecutive segments:
 *   S = S0 (NULL: zero); for d = 0..P-1: S_in[d] = S, S = Diag(exp(log_Gamma[d])) S + S_star[d];
 *   S_T = S.
 * log_Gamma: device float[P,B,H,dk]; S_star: device float[P,B,H,dk,dv] (pair d
 * at index d, in sequence order); S0: device float[B,H,dk,dv] or NULL; S_in:
 * device float[P,B,H,dk,dv] or NULL; S_T: device float[B,H,dk,dv] or NULL (one
 * of the two outputs must be given). Segment d's own S_in is the S_T of a
 * call with the first d pairs (P = d; P = 0 copies S0, or writes zeros).
 * S_in may be S_star exactly and S_T may be S0 exactly; no other overlap.
 * Asynchronous on `stream`.
 */
gla_status gla_pair_scan(int P, const float* log_Gamma, const float* S_star, const float* S0, float* S_in,
                         float* S_T, int B, int H, int dk, int dv, cudaStream_t stream);

/*
 * gla_pair_combine — in place, (log_Gamma1, S1) <- (log_Gamma2, S2) o (log_Gamma1, S1):
 *   S1 = Diag(exp(log_Gamma2)) S1 + S2,  log_Gamma1 = log_Gamma2 + log_Gamma1,
 * where pair 1 is the earlier segment. Device float[B,H,dk] and float[B,H,dk,dv]
 * each; pair 2 is not written and may not overlap pair 1. Asynchronous on `stream`.
 */
gla_status gla_pair_combine(const float* log_Gamma2, const float* S2, float* log_Gamma1, float* S1,
                            int B, int H, int dk, int dv, cudaStream_t stream);

/*
 * gla_bwd — the backward pass: gradients of a scalar loss L through the
 * forward pass described by the same inputs, given grad_O = dL/dO and
 * grad_ST = dL/dS_T (NULL: zero). It returns dL/dq, dL/dk, dL/dv, dL/dlog_g
 * (shaped like log_g: per key, per token, or per head summed over batch
 * rows) and dL/dS0 (even when S0 is NULL, i.e. zero). The chunkwise form
 * follows the GLA paper's §3.3 / §4.2: a forward sweep keeps the state
 * entering every chunk, a reverse sweep carries dL/dS through the chunks, and
 * the gate gradient is the reverse cumulative sum over tokens of
 * q (.) dq - k (.) dk (plus rowsum(grad_ST (.) S_T) at the last token).
 * Every gate mode and both dtypes are supported (q, k, v and grad_O in
 * `dtype`; all gradients fp32; dk <= 256). Three forms compute it:
 *   chunk form (AUTO's choice for bf16 inputs with dk in {128, 256}, dv a
 *     multiple of 128, q, k, v and grad_O 16-byte aligned, and any gate but
 *     the bilinear one; also GLA_PATH_TENSOR, which returns
 *     GLA_ERR_UNSUPPORTED for other inputs): 64-row chunks on the tcgen05
 *     tensor cores. The chunk pass's state sweeps keep every chunk's state
 *     and every chunk's dL/dS (bf16), then one chunk-parallel kernel forms
 *     dq, dk, dv and the gate terms. bf16 operands, fp32 accumulation, like
 *     the forward pass.
 *   split form (AUTO's choice for the other bf16 inputs with dk in
 *     {64, 128, 256} and no bilinear gate; GLA_PATH_SPLIT): 16-row chunks
 *     whose products run on the tensor cores (mma.sync) with every
 *     non-input operand split into hi + lo bf16 parts, about 16 mantissa
 *     bits, fp32 accumulation.
 *   CUDA-core form (fp32 inputs, other shapes, the bilinear gate, or
 *     GLA_PATH_SIMT): 16-row chunks in fp32 on CUDA cores.
 * The bilinear gate takes log_b and returns dL/dlog_b in grad_log_b
 * ([B,H,T,dv], may be NULL), on the CUDA-core form; that gradient is the
 * reverse cumulative sum over tokens of o (.) do - v (.) dv (plus
 * colsum(grad_ST (.) S_T) at the last token), with o recomputed inside.
 * (The backward is the next step after the forward pass; no page gives
 * numbers for it.)
 *
 * Ownership and asynchrony are as for gla_fwd_ex: every pointer is a device
 * pointer owned by the caller, work is enqueued on `stream`, and the caller
 * supplies a workspace of gla_bwd_workspace_size(p) bytes (256-byte aligned;
 * the size depends on the form the pointers and shapes select: the chunk
 * form keeps two bf16 states per 64-row chunk, BH * ceil(T/64) * dk * dv * 4
 * bytes in all, the 16-row forms one fp32 state per 16-row chunk and
 * per-tile partial gradients). grad_log_g and grad_S0 may be NULL (not
 * wanted); grad_log_g must be NULL without a gate. Outputs may not overlap
 * inputs or each other. Results are bitwise reproducible.
 */
typedef struct {
    const void* q;          /* [B,H,T,dk] dtype */
    const void* k;          /* [B,H,T,dk] dtype */
    const void* v;          /* [B,H,T,dv] dtype */
    const float* log_g;     /* as in gla_fwd_params */
    const float* S0;        /* [B,H,dk,dv] or NULL */
    const void* grad_O;     /* [B,H,T,dv] dtype */
    const float* grad_ST;   /* [B,H,dk,dv] or NULL */
    float* grad_q;          /* [B,H,T,dk] */
    float* grad_k;          /* [B,H,T,dk] */
    float* grad_v;          /* [B,H,T,dv] */
    float* grad_log_g;      /* shaped like log_g, or NULL */
    float* grad_S0;         /* [B,H,dk,dv] or NULL */
    int B, H, T, dk, dv;
    gla_dtype dtype;
    gla_gate gate;
    void* workspace;
    size_t workspace_bytes;
    int path;               /* gla_path: AUTO, TENSOR (chunk form), SPLIT or SIMT (see above) */
    const float* log_b;     /* [B,H,T,dv] log(beta_t) for GLA_GATE_BILINEAR, else NULL */
    float* grad_log_b;      /* [B,H,T,dv] dL/dlog_b, or NULL (not wanted; bilinear gate only) */
} gla_bwd_params;

gla_status gla_bwd(const gla_bwd_params* p, cudaStream_t stream);

/* Bytes of workspace gla_bwd needs for *p (0 for invalid parameters). */
size_t gla_bwd_workspace_size(const gla_bwd_params* p);

/* gla_bwd in its stages, for timing each kernel: gla_bwd(p) ==
 * gla_bwd_stage(p, 0) ... gla_bwd_stage(p, n-1) on one stream (each stage
 * reads what the ones before it wrote to the workspace). The chunk form has
 * up to six (gate prep, state sweep, dL/dS sweep, boundary term, gradients,
 * gate tail); the 16-row forms one. gla_bwd_num_stages returns n, or -1 for
 * invalid parameters; gla_bwd_stage_name a static string naming stage i's
 * kernel ("invalid" out of range). */
int gla_bwd_num_stages(const gla_bwd_params* p);
gla_status gla_bwd_stage(const gla_bwd_params* p, int stage, cudaStream_t stream);
const char* gla_bwd_stage_name(const gla_bwd_params* p, int stage);

/* Synchronises `stream`, then reads and clears the library's device status
 * word for the current device. GLA_ERR_TIMEOUT if a kernel gave up on a
 * bounded wait since the last call, GLA_ERR_CUDA if the stream reports an
 * error, else GLA_OK. */
gla_status gla_device_status(cudaStream_t stream);

/*
 * gla_selftest_bounded_wait — exercises the failure path of the kernels'
 * bounded waits without faulting anything. (No counterpart in the papers: a
 * diagnostic.) Enqueues on `stream` a one-warp kernel that waits, with the
 * same bounded mbarrier wait the pipelined kernels use, on a shared-memory
 * barrier. With arrive = 0 nothing ever arrives: after limit_us microseconds
 * the wait gives up, the kernel records a timeout in the device status word
 * and returns, so the next gla_device_status() reports GLA_ERR_TIMEOUT and the
 * context stays usable. With arrive != 0 the kernel arrives on the barrier
 * first and the wait succeeds at once. The kernel holds no tensor memory and
 * issues no asynchronous copy. limit_us must be in 1..1000000, else
 * GLA_ERR_INVALID_ARG.
 */
gla_status gla_selftest_bounded_wait(unsigned limit_us, int arrive, cudaStream_t stream);

/* A static, human-readable name for s. */
const char* gla_status_string(gla_status s);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int gla_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GLA_H_ */
