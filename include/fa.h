/*
 * fa.h -- C ABI of libfa.so: exact IO-aware attention (forward with log-sum-exp, and the
 * recompute-based backward) for NVIDIA GB300 (sm_103a).
 *
 * Operation (the plain definition; the kernels reach it up to rounding order):
 *   S = scale * Q K^T,  P = softmax(S) row-wise,  O = P V,  LSE_i = ln sum_j exp(S_ij)
 *   -- "FlashAttention: from IO-Aware Attention to GPU work partitioning"
 *      (blog.euler0525.cn), sections "Attention 的性能瓶颈" (S, P, O) and "FlashAttention-2"
 *      (L_i = m_i + log l_i); "15. FlashAttention" (inference.shantanugoel.com), sections
 *      "Online softmax: normalize as you go" and "The algorithm in plain PyTorch".
 *   With causal != 0, key j is visible to query i iff j <= i (query and key sequences
 *   have the same length N), as in blog.euler0525.cn, section "Tile Size 与 Causal
 *   Attention" (S_ij = -inf for j > i).
 *
 * Layout: Q, K, V, O, dO, dQ, dK, dV are bf16, contiguous row-major [B, H, N, d]
 * (element (b,h,n,e) at ((b*H + h)*N + n)*d + e). LSE is fp32 [B, H, N], natural log of
 * the scaled scores. Every pointer is a device pointer unless stated otherwise.
 *
 * Ownership: the caller owns every buffer; the library keeps no state between calls
 * besides one device error word per device (see fa_device_error).
 *
 * Execution: calls only enqueue work on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and return; they never synchronise. FA_OK means the launch was accepted;
 * device-side faults surface at the caller's next synchronisation. A kernel that waits
 * on an internal barrier for longer than a few seconds gives up, records an error code
 * in the device error word and exits without faulting.
 *
 * Errors: arguments are checked on the host before anything is launched; a call that
 * returns an error has launched nothing.
 *   FA_ERR_INVALID_ARG  null pointer (when there is work), negative B/H/N, causal not 0/1,
 *                       scale not finite or not > 0, workspace too small
 *   FA_ERR_UNSUPPORTED  d not 64 or 128; sizes beyond the int32 range of the kernels
 *   FA_ERR_ALIGNMENT    a bf16 tensor not 16-byte aligned, LSE not 4-byte aligned,
 *                       workspace not 256-byte aligned (TMA needs 16-byte bases)
 *   FA_ERR_CUDA         a CUDA runtime/driver call failed (fa_last_cuda_error gives it)
 * B*H*N == 0 is valid: nothing is launched and FA_OK is returned.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,
    FA_ERR_UNSUPPORTED = 2,
    FA_ERR_ALIGNMENT = 3,
    FA_ERR_CUDA = 4,
    FA_ERR_TIMEOUT = 5
} fa_status;

/*
 * Forward: O = softmax(scale Q K^T) V and LSE, computed tile by tile with the online-softmax
 * recurrence (running max m, running sum l, rescale alpha = exp(m_old - m_new) applied to l
 * and to the unnormalised accumulator; O = acc / l at the end; LSE = m + ln l), so the N x N
 * matrices never reach HBM ("15. FlashAttention", section "Online softmax: normalize as you
 * go"; blog.euler0525.cn, section "FlashAttention-2").
 *   q, k, v  in : bf16 [B,H,N,d]
 *   o        out: bf16 [B,H,N,d]
 *   lse      out: fp32 [B,H,N]  (natural log, of scale * q.k)
 *   d in {64, 128}; causal in {0, 1}; scale > 0 (1/sqrt(d) for standard attention).
 */
fa_status fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, int causal, float scale, struct CUstream_st* stream);

/*
 * Forward with grouped KV heads, a query offset and an optional sliding window ("15.
 * FlashAttention", inference.shantanugoel.com, sections "The algorithm in plain PyTorch" and
 * "Details worth noticing": query head h reads KV head h / (Hq / Hkv); query row i sits at
 * absolute position Tk - Tq + i, so the newest query lines up with the newest key and one call
 * serves prefill (Tq = Tk), chunked prefill (Tq < Tk) and decode (Tq = 1); section "Stretch
 * exercises", item 3: a window of W keeps only keys at positions >= position - W).
 * Key j is visible to query row i, at position p = Tk - Tq + i, iff
 *     (causal == 0 || j <= p)  and  (window < 0 || j >= p - window).
 *   q        in : bf16 [B,Hq,Tq,d]      k, v in : bf16 [B,Hkv,Tk,d]
 *   o        out: bf16 [B,Hq,Tq,d]      lse  out: fp32 [B,Hq,Tq]
 *   Hq % Hkv == 0 (Hkv = Hq: multi-head; Hkv = 1: multi-query).
 *   window = -1 for none; window >= 0 requires causal = 1 (the window is measured back from the
 *   diagonal). Every query row must see a key: Tk >= 1, and with causal Tq <= Tk; otherwise
 *   FA_ERR_INVALID_ARG. Other arguments and errors as fa_forward, which is this call with
 *   Hq = Hkv = H, Tq = Tk = N, window = -1. B*Hq*Tq == 0 launches nothing.
 *   With grouped heads and Tq <= 64 (decode, short chunks) the query heads of a KV head are
 *   processed as one block of (Hq / Hkv) * Tq rows, so each KV head's K and V are read once
 *   for the whole group; the results are the same.
 */
fa_status fa_forward_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int Hq, int Hkv, int Tq, int Tk, int d, int causal, int window,
                        float scale, struct CUstream_st* stream);

/*
 * Split-KV forward ("flash-decoding"; "15. FlashAttention", inference.shantanugoel.com, section
 * "Decode is different: flash-decoding"). Same operation, arguments and results as
 * fa_forward_ex, but every query block's visible key range is cut into `nsplit` chunks that
 * run as separate work units, so short query blocks (decode, small B*Hq*Tq) still fill the
 * GPU. Each chunk writes its partial result -- the chunk's normalised O_s (fp32) and
 * LSE_s = m_s + ln l_s, or LSE_s = -inf for a row that sees no key of the chunk -- and a
 * second kernel merges them by the page's rule m = max m_s, l = sum e^(m_s - m) l_s,
 * a = sum e^(m_s - m) a_s, O = a / l (with normalised partials: O = sum_s e^(LSE_s - LSE) O_s,
 * LSE = ln sum_s e^LSE_s). Results equal fa_forward_ex's up to rounding order.
 *   nsplit    1 .. FA_MAX_SPLITS; 1 is fa_forward_ex (no workspace used).
 *   workspace device buffer of >= fa_forward_splitkv_workspace_bytes(B, Hq, Tq, d, nsplit)
 *             bytes, 256-byte aligned, or NULL (allocated and freed on `stream`).
 * Errors as fa_forward_ex; nsplit out of range -> FA_ERR_INVALID_ARG.
 */
#define FA_MAX_SPLITS 64

size_t fa_forward_splitkv_workspace_bytes(int B, int Hq, int Tq, int d, int nsplit);

/*
 * A key-split count for fa_forward_splitkv on these sizes and `num_sms` SMs (1: no split):
 * the library's cost model, in 128-key tile steps, of rounds of (key chunk + fixed per-unit
 * cost) plus the merge; a split is chosen only when it is clearly cheaper than the unsplit
 * launch. Pure host logic (no device access). Returns 1 for invalid sizes.
 */
int fa_forward_choose_splits(int B, int Hq, int Hkv, int Tq, int Tk, int num_sms);

fa_status fa_forward_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
                             int window, float scale, int nsplit, void* workspace,
                             struct CUstream_st* stream);

/*
 * Bytes of device workspace fa_backward needs for these sizes: two 16-byte records per query
 * row holding -LSE/scale and -D_i (D_i = O_i . dO_i) as exact three-part bf16 sums, [B*H, Npad]
 * each, an fp32 dQ accumulator of B*H*Npad*d elements (Npad = N rounded up to 128) and 256 bytes for
 * the counter that hands out the main kernel's work units. In total B*H*Npad*(32 + 4d) + 256
 * bytes. Returns 0 for invalid sizes or when B*H*N == 0.
 */
size_t fa_backward_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward by recomputation: rebuilds S and P = exp(S - LSE) tile by tile from Q, K, V and
 * the saved LSE, then dV = P^T dO, dP = dO V^T, D_i = O_i . dO_i, dS = P (.) (dP - D),
 * dQ = scale dS K, dK = scale dS^T Q (blog.euler0525.cn, sections "Tiling、Fusion 与
 * Backward Recomputation" and "FlashAttention-2"; the scale factor on dQ and dK follows from
 * the chain rule through S = scale Q K^T). dQ partial sums from different key tiles are
 * added in fp32 (section "Sequence Parallelism": column-oriented partition with atomic add).
 *   q, k, v, o, dout in : bf16 [B,H,N,d];  lse in : fp32 [B,H,N] from fa_forward
 *   dq, dk, dv       out: bf16 [B,H,N,d]
 *   workspace: device buffer of >= fa_backward_workspace_bytes(B,H,N,d) bytes, 256-byte
 *              aligned, used for the duration of the call's work on `stream`; or NULL, in
 *              which case the library allocates and frees it on `stream` (cudaMallocAsync).
 */
fa_status fa_backward(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                      int H, int N, int d, int causal, float scale, void* workspace,
                      struct CUstream_st* stream);

/*
 * Backward of fa_forward_ex (same visibility rule and shapes): dq bf16 [B,Hq,Tq,d]; dk, dv
 * bf16 [B,Hkv,Tk,d], where the gradient of a KV head sums the contributions of all Hq / Hkv
 * query heads that read it. Keys no query sees get zero gradient; with B*Hq*Tq == 0 and
 * B*Hkv*Tk > 0 the call only zeroes dk and dv (q, k, v, o, lse, dout, dq may then be NULL).
 *   workspace: >= fa_backward_workspace_bytes(B, Hq, Tq, d) bytes, 256-byte aligned, or NULL
 *              (allocated and freed on `stream`).
 * Errors as fa_forward_ex and fa_backward. fa_backward is this call with Hq = Hkv = H,
 * Tq = Tk = N, window = -1.
 */
fa_status fa_backward_ex(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                         int Hq, int Hkv, int Tq, int Tk, int d, int causal, int window,
                         float scale, void* workspace, struct CUstream_st* stream);

/*
 * Allocation-free backward (no counterpart in the pages: an integration convenience).
 *
 * Same computation, arguments and results as fa_backward, for callers that may not allocate
 * device memory at call time: runtimes that plan every device buffer once at start-up and
 * forbid allocation afterwards, hosts embedding the library without access to an allocator,
 * or loops where an allocation's latency or fragmentation is not acceptable. Instead of a
 * caller buffer or cudaMallocAsync, the workspace is one file-scope device array of
 * FA_NOALLOC_SCRATCH_BYTES bytes inside libfa.so, which every GPU that loads the library keeps
 * until the process exits. This call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).
 *   - Sizes whose workspace (fa_backward_workspace_bytes) exceeds FA_NOALLOC_SCRATCH_BYTES are
 *     rejected with FA_ERR_UNSUPPORTED before anything is launched (for example B*H = 64,
 *     N = 2048, d = 64 needs 37.7 MB and fits; B*H = 64, N = 4096, d = 128 needs 143 MB and
 *     does not). Other argument errors are those of fa_backward.
 *   - The first call on a device looks up the array's device address (with that device
 *     current) and caches it; make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents; the kernels
 *     initialise every part of it they read, so no clearing is needed. Calls whose work
 *     overlaps on the GPU (different streams, or different host threads, without ordering
 *     between them) race on the array: order them.
 */
#define FA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

fa_status fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, int causal, float scale,
                              struct CUstream_st* stream);

/* FA_NOALLOC_SCRATCH_BYTES as compiled into this libfa.so: the size of the workspace array
 * fa_backward_noalloc uses (a binding can read it instead of repeating the macro). */
size_t fa_noalloc_scratch_bytes(void);

/*
 * One forward + backward step on host-resident tensors (no counterpart in the pages: an
 * integration convenience for callers whose activations live in host memory). Copies Q, K, V
 * and dO to the device, runs fa_forward_ex and then fa_backward_ex on them, and copies O, LSE,
 * dQ, dK and dV back. The KV heads, flattened over the batch, are cut into `nchunks` chunks
 * of nearly equal size, each with the query heads that read them. Every chunk's copies in, its
 * two kernels and its copies out (O and LSE once its forward is done, the gradients after its
 * backward) go to internal streams -- one for copies in, two for kernels, one for copies out --
 * so that one chunk's copies overlap other chunks' kernels. Results equal those of
 * fa_forward_ex and fa_backward_ex on the same inputs (dQ up to the order in which its fp32
 * partial sums are added).
 *   q, dout in : host bf16 [B,Hq,Tq,d];  k, v in : host bf16 [B,Hkv,Tk,d]
 *   o out : host bf16 [B,Hq,Tq,d];  lse out : host fp32 [B,Hq,Tq]
 *   dq out: host bf16 [B,Hq,Tq,d];  dk, dv out: host bf16 [B,Hkv,Tk,d]
 *   Host buffers should be page-locked (cudaHostAlloc or cudaHostRegister) for the copies to
 *   overlap with the kernels; pageable memory gives the same results without the overlap.
 *   nchunks: 1 .. FA_MAX_HOST_CHUNKS, or 0 for the library's choice (4); a value above B*Hkv
 *            is reduced to B*Hkv.
 *   device_buffer: >= fa_forward_backward_host_device_bytes(B, Hq, Hkv, Tq, Tk, d, nchunks)
 *            bytes of device memory, 256-byte aligned, used until the step is done on
 *            `stream`; or NULL, in which case the library allocates and frees it on `stream`
 *            (cudaMallocAsync).
 *   stream: the step starts after the work queued on `stream` before the call, and work
 *           queued on `stream` after the call starts once the step, copies out included, is
 *           done. As with cudaMemcpyAsync, the host buffers must stay valid and unmodified
 *           until then. Calls from several host threads are serialised while they enqueue.
 * Errors as fa_forward_ex and fa_backward_ex; FA_ERR_INVALID_ARG for a NULL tensor pointer
 * where that tensor has elements, or nchunks outside 0 .. FA_MAX_HOST_CHUNKS.
 */
#define FA_MAX_HOST_CHUNKS 16

/* Device bytes fa_forward_backward_host needs (0 for invalid arguments). */
size_t fa_forward_backward_host_device_bytes(int B, int Hq, int Hkv, int Tq, int Tk, int d,
                                             int nchunks);

fa_status fa_forward_backward_host(const void* q, const void* k, const void* v, const void* dout,
                                   void* o, float* lse, void* dq, void* dk, void* dv, int B,
                                   int Hq, int Hkv, int Tq, int Tk, int d, int causal, int window,
                                   float scale, int nchunks, void* device_buffer,
                                   struct CUstream_st* stream);

/*
 * Row softmax of naive (materialised) attention -- the comparison point the IO-aware method is
 * measured against, not part of it ("15. FlashAttention", section "The score matrix is the
 * problem" and "Stretch exercises" item 1; "FlashAttention V1", the standard-attention
 * baseline). A GEMM writes the full score matrix to HBM; this call reads it back and writes
 * the probabilities and the row log-sum-exp; a second GEMM forms O = P V.
 *   s    in : fp32 [rows, N], rows = B*H*N, raw dot products q_i . k_j of each head
 *   p    out: bf16 [rows, N], P_ij = exp(scale s_ij - m_i) / l_i for visible j, else 0
 *   lse  out: fp32 [rows],   m_i + ln l_i (natural log of the scaled scores)
 *   With causal = 1, row r sees keys j <= r mod N. Safe softmax (max subtracted), fp32.
 * Errors: FA_ERR_INVALID_ARG (negative sizes, causal not 0/1, scale not finite or not > 0,
 * NULL pointers with work), FA_ERR_ALIGNMENT, FA_ERR_CUDA. rows * N == 0 launches nothing.
 */
fa_status fa_naive_softmax(const float* s, void* p, float* lse, long long rows, int N, int causal,
                           float scale, struct CUstream_st* stream);

/*
 * Diagnostic of the failure path (no counterpart in the pages). Launches one warp that waits,
 * through the same bounded mbarrier wait the attention kernels use, on a barrier nothing ever
 * arrives on; after `limit_us` microseconds (1 .. 1000000) the wait gives up, records code 1
 * (load) in the device error word and the kernel returns, leaving the context usable. Read the
 * code with fa_device_error. Nothing faults or hangs.
 */
fa_status fa_selftest_wait_timeout(unsigned int limit_us, struct CUstream_st* stream);

/* Human-readable name of a status code (static string). */
const char* fa_status_string(fa_status s);

/* The cudaError_t of the last FA_ERR_CUDA returned on this thread (0 if none). */
int fa_last_cuda_error(void);

/*
 * Synchronises `stream`, then reads and clears this device's error word. *code receives 0
 * when no kernel gave up on a wait since the last call, else the first error code
 * (1 load, 2 MMA completion, 3 buffer release, 4 softmax signal). Returns FA_ERR_TIMEOUT
 * when *code != 0, FA_ERR_CUDA if synchronisation or the read failed, else FA_OK.
 */
fa_status fa_device_error(struct CUstream_st* stream, int* code);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
