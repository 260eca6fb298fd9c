/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 library: the forward
 * pass (the hot path), its key-split form, the backward pass and an FP8 forward.
 *
 * The library computes, for bf16 tensors in [batch, seq, heads, d_head]
 * layout (the layout of the input generator on "Flash Attention 2 Chapter2",
 * section on mapping attention tensors to mma operands),
 *
 *     O[b,i,h,:]  = sum_j softmax_j(scale * q_i . k_j) * v_j        (bf16 out)
 *     LSE[b,h,i]  = log sum_j exp(scale * q_i . k_j)                (fp32, natural log)
 *
 * "GPU 内核与 FlashAttention" §10 defines S, P and O; §11.3 the online softmax
 * recurrence the kernel uses; §13.2 and §14.1 the per-row log-sum-exp kept by
 * the forward pass.  "Flash Attention实现深度解析" §3.1 gives the host entry
 * that returns {out, softmax_lse} with lse shaped [batch, heads, max_seqlen_q]
 * and packed [total, heads, d_head] tensors for variable-length batches.
 *
 * Conventions shared by every entry point
 *   - Pointers named q, k, v, o, lse, cu_seqlens* are DEVICE pointers owned by
 *     the caller.  The library never allocates global memory per call and never
 *     frees caller memory.  Tensor memory (TMEM) is allocated and released
 *     inside each kernel.
 *   - q, k, v, o must be 16-byte aligned and densely packed (no padding).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work and return; results are valid once the stream is
 *     synchronised.  Errors detected on the device (timeouts, inconsistent
 *     cu_seqlens) are reported by fa_check_status().
 *   - Return value: FA_OK (0) or one of the negative FA_ERR_* codes.  Argument
 *     errors are detected on the host before anything is enqueued.
 *   - Not thread-safe with respect to fa_set_* / fa_autotune, which change
 *     process-wide settings.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

#define FA_OK 0
#define FA_ERR_INVALID_ARG (-1)  /* null pointer, negative size, bad scale, B*H too large */
#define FA_ERR_UNSUPPORTED (-2)  /* d_head not in {64, 128} (FP8: not 128), or no sm_103a
                                    device, or the device's shared-memory window does not
                                    fit the backward kernel's layout (fa_check_status)   */
#define FA_ERR_ALIGN (-3)        /* a tensor pointer is not 16-byte aligned             */
#define FA_ERR_CUDA (-4)         /* a CUDA call failed; fa_last_cuda_error() has it     */
#define FA_ERR_TIMEOUT (-5)      /* a device-side wait gave up (fa_check_status)        */
#define FA_ERR_NO_DEVICE (-6)    /* no CUDA device is visible                           */
#define FA_ERR_BAD_SEQLENS (-7)  /* cu_seqlens inconsistent with the maximum lengths    */
#define FA_ERR_SCRATCH_LIMIT (-8) /* problem needs more than the fixed 16 MiB scratch   */

/*
 * fa_fwd -- attention forward, self-attention shapes (Nq = Nk = N).
 *
 * Dense form (cu_seqlens == NULL):
 *   q, k, v, o : bf16 [B, N, H, d], contiguous; element (b, n, h, c) at
 *                ((b * N + n) * H + h) * d + c.
 *   lse        : fp32 [B, H, N].
 * Variable-length form (cu_seqlens != NULL):
 *   cu_seqlens : int32 [B + 1] device array, cu[0] = 0, non-decreasing; sequence
 *                b owns packed rows [cu[b], cu[b+1]) of q, k, v and o, each
 *                [total, H, d] with total = cu[B].  Sequences attend only within
 *                themselves.
 *   N          : the maximum sequence length (every length must be <= N); it
 *                bounds the launch grid and is the row stride of lse.
 *   lse        : fp32 [B, H, N]; entries (b, h, i) with i >= len(b) are not written.
 *   A sequence longer than N is reported as FA_ERR_BAD_SEQLENS by
 *   fa_check_status(), and its CTAs write nothing.
 * scale        : softmax scale, finite and > 0 (1/sqrt(d) is the usual value).
 * d            : 64 or 128.
 * B == 0 or N == 0 is a no-op that returns FA_OK.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int N, int H,
           int d, float scale, const int* cu_seqlens, void* stream);

/*
 * fa_fwd_qk -- general form with separate query and key lengths (for example
 * the 64-query by 4096-key slice of "Flash Attention 2 Chapter2", introduction).
 *
 * Dense form (both cu pointers NULL): q, o [B, Nq, H, d]; k, v [B, Nk, H, d];
 *   lse [B, H, Nq].  Nk must be >= 1 when Nq >= 1.
 * Variable-length form (both cu pointers non-NULL): q, o [total_q, H, d];
 *   k, v [total_k, H, d]; Nq / Nk are the maximum query / key lengths.  A
 *   sequence with no keys gets o = 0 and lse = -inf (log of an empty sum).
 * Passing exactly one cu pointer is FA_ERR_INVALID_ARG.
 */
int fa_fwd_qk(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Nq,
              int Nk, int H, int d, float scale, const int* cu_seqlens_q,
              const int* cu_seqlens_k, void* stream);

/*
 * fa_fwd_ex -- the general entry: fa_fwd_qk plus grouped key/value heads and
 * flags.
 *   Hk    : key/value heads; H must be a multiple of Hk.  Query head h reads
 *           key/value head h / (H / Hk) ("GPU 内核与 FlashAttention" §14.2,
 *           MQA / GQA).  k and v are [B, Nk, Hk, d] (dense) or
 *           [total_k, Hk, d] (variable length); q, o and lse are as in fa_fwd_qk.
 *   flags : 0, or FA_FLAG_CAUSAL for the causal mask of §14.4, aligned
 *           bottom-right when the lengths differ: query i sees keys
 *           j <= i + (Nk - Nq) (per sequence in the variable-length form).
 *           Key tiles above the diagonal are skipped.  Rows that see no key
 *           get o = 0 and lse = -inf.
 * Unknown flag bits, Hk <= 0 or H % Hk != 0 give FA_ERR_INVALID_ARG.
 */
#define FA_FLAG_CAUSAL 1
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Nq,
              int Nk, int H, int Hk, int d, float scale, const int* cu_seqlens_q,
              const int* cu_seqlens_k, int flags, void* stream);

/*
 * Key-split form for short query sets (dense tensors; for example the
 * 64-query x 4096-key slice of "Flash Attention 2 Chapter2", introduction).
 * The key range of every (batch, head, 256-row query block) is cut into
 * num_splits contiguous ranges that run on different SMs; each writes its
 * normalised fp32 output and log-sum-exp to `workspace`, and a second kernel
 * merges them exactly ("GPU 内核与 FlashAttention" §11.2: LSE = log sum_s
 * e^LSE_s, O = sum_s e^(LSE_s - LSE) O_s).
 *
 * fa_splitkv_num_splits      -- splits a call with these sizes would use for
 *                               `requested` (<= 0: chosen to give every SM a
 *                               unit, at least two key tiles per split; capped
 *                               at 128 and at the number of 128-key tiles).
 *                               Needs the current device; returns the count or
 *                               a negative FA_ERR_* code.
 * fa_splitkv_workspace_bytes -- bytes of workspace for num_splits splits:
 *                               num_splits * B * H * Nq * (d + 1) * 4; negative
 *                               FA_ERR_* code on bad arguments.
 * fa_fwd_splitkv             -- arguments as fa_fwd_ex (dense only, no
 *                               cu_seqlens), plus num_splits (<= 0: choose) and
 *                               a caller-owned DEVICE workspace, 16-byte aligned,
 *                               of at least fa_splitkv_workspace_bytes(...,
 *                               fa_splitkv_num_splits(...)) bytes; a smaller or
 *                               misaligned workspace gives FA_ERR_INVALID_ARG.
 *                               The workspace is fully rewritten by every call;
 *                               calls that share one must not overlap on the GPU.
 */
int fa_splitkv_num_splits(int B, int Nq, int Nk, int H, int d, int requested);
long long fa_splitkv_workspace_bytes(int B, int Nq, int H, int d, int num_splits);
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Nq,
                   int Nk, int H, int Hk, int d, float scale, int flags, int num_splits,
                   void* workspace, unsigned long long workspace_bytes, void* stream);

/*
 * fa_fwd_splitkv_noalloc -- the key-split forward (fa_fwd_splitkv) for callers
 * that cannot allocate device memory when attention runs: runtimes that reserve
 * all device memory up front and forbid later allocations, real-time paths
 * where an allocation's latency or failure is not acceptable, or C callers
 * with no memory pool of their own.  The pages have no counterpart; this is a
 * deployment variant of the same computation.
 *   Arguments as fa_fwd_splitkv without the workspace: the caller passes only
 *   inputs and outputs (device pointers), and nothing is allocated.
 *   Scratch: a fixed 16 MiB array inside the library, held on every GPU that
 *   loads the library until the process exits.  A problem needing more
 *   (B * H * Nq * splits * (d + 1) * 4 bytes, splits from
 *   fa_splitkv_num_splits) returns FA_ERR_SCRATCH_LIMIT and launches nothing.
 *   The first call on a device looks up the array's device address (a one-time
 *   set-up per device); make that first call before any stream capture.
 *   All calls on a device share the array: calls that overlap on the GPU (other
 *   streams or host threads) race and must be serialised by the caller.  No
 *   part of the array needs clearing: each call writes every entry it reads.
 *   The array used is the one of the CURRENT device: `stream` must belong to
 *   it (a stream of another device gives FA_ERR_INVALID_ARG).
 *   Argument errors are those of fa_fwd_splitkv, checked in the same order
 *   (for example d not in {64, 128} is FA_ERR_UNSUPPORTED).
 *   If fa_check_status() then reports an error (a device wait gave up), o and
 *   lse of that call are undefined: the merge may have combined partial
 *   results that the aborted kernel never wrote with entries an earlier call
 *   left in the shared array.
 */
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                           int Nq, int Nk, int H, int Hk, int d, float scale, int flags,
                           int num_splits, void* stream);

/*
 * fa_check_status -- synchronises `stream`, then returns and clears the first
 * device-side error recorded since the last call (FA_OK if none).  When
 * `info` is not NULL it receives {flat block index, warp, wait site} of that
 * error (zeros if none).  Returns FA_ERR_CUDA if synchronisation fails.
 * After a non-OK status the outputs of the calls since the previous check are
 * undefined (a kernel that gave up stops early and leaves rows unwritten).
 */
int fa_check_status(void* stream, int* info);

/* Human-readable text for an FA_* code (static storage). */
const char* fa_strerror(int code);

/* The cudaError_t of the most recent FA_ERR_CUDA on this thread. */
int fa_last_cuda_error(void);

/*
 * Backward pass ("GPU 内核与 FlashAttention" §13.2, FlashAttention-2's blockwise
 * backward): gradients of O = softmax(scale * Q K^T) V with respect to q, k
 * and v, given dout = dLoss/dO, the forward's output o and its log-sum-exp.
 *   q, o, dout, dq : [B, Nq, H, d] bf16, contiguous
 *   k, v, dk, dv   : [B, Nk, Hk, d] bf16, contiguous (H a multiple of Hk; the
 *                    key/value gradients of the H/Hk query heads sharing a
 *                    key/value head are summed, §14.2)
 *   lse            : [B, H, Nq] fp32, natural log, as written by the forward
 *                    with the same flags (rows with lse = -inf get no gradient)
 *   flags          : 0 or FA_FLAG_CAUSAL (the forward's mask)
 *   workspace      : device memory of at least fa_bwd_workspace_bytes(B, Nq, H,
 *                    d) bytes, 16-byte aligned, owned by the caller; fully
 *                    overwritten (the fp32 dQ accumulator, D = rowsum(dO o O)
 *                    and the scaled log-sum-exp), nothing needs to persist.
 * d = 64 or 128 (FA_ERR_UNSUPPORTED otherwise); dense tensors (packed ones: fa_bwd_varlen).  Three
 * kernels are enqueued on `stream`: preprocessing (D and a cleared
 * accumulator), the key-block kernel (writes dk, dv; adds dQ into the
 * accumulator) and the conversion of the accumulator to bf16 dq.  Errors as
 * fa_fwd_ex; FA_ERR_INVALID_ARG also for a missing or short workspace.
 * B = 0 or H = 0 (or Nq = Nk = 0) is a no-op; Nq > 0 with Nk = 0 is
 * FA_ERR_INVALID_ARG as in the forward; Nq = 0 writes dk = dv = 0.
 * fa_bwd_workspace_bytes returns the size, or a negative FA_* code.
 */
long long fa_bwd_workspace_bytes(int B, int Nq, int H, int d);
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int Nq, int Nk, int H, int Hk,
           int d, float scale, int flags, void* workspace, long long workspace_bytes, void* stream);

/*
 * Variable-length backward: the same gradients for packed sequences, as the
 * forward's variable-length form lays them out ([FMHA] §3.1): q, o, dout, dq
 * are [total_q, H, d], k, v, dk, dv [total_k, Hk, d] (rows of sequence b at
 * cu_seqlens[b] .. cu_seqlens[b + 1] - 1), lse [B, H, max_seqlen_q] as the
 * variable-length forward writes it.  cu_seqlens_q / cu_seqlens_k: device
 * int32 [B + 1], non-decreasing from 0, 4-byte aligned; every length at most
 * the given maximum (a longer one is reported as FA_ERR_BAD_SEQLENS by
 * fa_check_status and its units write nothing).  The workspace is
 * fa_bwd_workspace_bytes(B, max_seqlen_q, H, d).  The causal mask is aligned
 * bottom-right within each sequence.  Rows of dq, dk, dv past the last
 * sequence are not written; a sequence without keys gets dq = 0.
 */
int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int B, int max_seqlen_q, int max_seqlen_k, int H, int Hk,
                  int d, float scale, int flags, void* workspace, long long workspace_bytes,
                  void* stream);

/*
 * FP8 forward ("GPU 内核与 FlashAttention" §15.5: e4m3 inputs with block
 * quantisation).  Quantisation: every block of values shares one fp32 scale
 * s = amax(block) / 448 (1 for an all-zero block) and a value x is stored as
 * the e4m3 code nearest to x / s (round to nearest even, saturating).
 * Blocks: 128 query rows of one head (Q), 128 keys of one key/value head (K),
 * one key/value head (V).  V is stored transposed.
 *
 * fa_fp8_sizes     -- sizes[0..5] = bytes of q8 [B, Nq, H, d], k8 [B, Nk, Hk, d],
 *                     vt8 [B, Hk, d, nk_pad] (nk_pad = Nk rounded up to 16),
 *                     and element counts of q_scale [B, H, ceil(Nq/128)],
 *                     k_scale [B, Hk, ceil(Nk/128)], v_scale [B, Hk] (fp32).
 * fa_quantize_fp8  -- fills those from bf16 q, k, v (layouts of fa_fwd_ex);
 *                     all device pointers, code buffers 16-byte aligned, scale
 *                     buffers 4-byte aligned (FA_ERR_ALIGN otherwise).  Reads
 *                     Q once and K, V twice (V's scale needs the whole head
 *                     before its codes); v_scale holds intermediate values until
 *                     the call's work on `stream` completes.
 * fa_fwd_fp8       -- the forward pass on them: o (bf16 [B, Nq, H, d]) and
 *                     lse (fp32 [B, H, Nq]) as fa_fwd_ex, scale the natural
 *                     softmax scale applied to the dequantised scores, flags 0
 *                     or FA_FLAG_CAUSAL.  S = Q K^T and O += P V run on the
 *                     tensor cores in e4m3 with fp32 accumulation; P is rounded
 *                     to e4m3 for the second product (the row sums use the
 *                     unrounded fp32 values).  Dense tensors (packed ones:
 *                     fa_fwd_fp8_varlen below), d = 128 only
 *                     (FA_ERR_UNSUPPORTED otherwise).
 */
int fa_fp8_sizes(int B, int Nq, int Nk, int H, int Hk, int d, long long* sizes);
int fa_quantize_fp8(const void* q, const void* k, const void* v, int B, int Nq, int Nk, int H, int Hk, int d,
                    void* q8, void* k8, void* vt8, float* q_scale, float* k_scale, float* v_scale, void* stream);
int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int B, int Nq, int Nk, int H, int Hk, int d, float scale,
               int flags, void* stream);

/*
 * Variable-length FP8 forward: packed sequences as in fa_fwd_ex's
 * variable-length form ("Flash Attention实现深度解析" §3.1), quantised per
 * sequence.
 *   cu_seqlens_q / cu_seqlens_k : device int32 [B + 1], 4-byte aligned,
 *       non-decreasing from 0; sequence b owns packed rows [cu[b], cu[b + 1]).
 *   total_q / total_k : packed rows of q / k (= cu[B]); max_seqlen_q / _k
 *       bound every length.  A sequence whose rows do not fit these bounds is
 *       reported as FA_ERR_BAD_SEQLENS by fa_check_status() (fa_fwd_fp8_varlen)
 *       and neither kernel touches memory for it.
 *   Blocks restart at every sequence: block j of sequence b is its rows
 *       128j .. 128j + 127 (Q: of one head; K: of one key/value head), and V has
 *       one block per (sequence, key/value head).  Scales are fp32
 *       q_scale [B, H, ceil(max_seqlen_q / 128)], k_scale [B, Hk,
 *       ceil(max_seqlen_k / 128)], v_scale [B, Hk]; blocks past a sequence's
 *       end get scale 1.
 *   Codes: q8 [total_q, H, d] and k8 [total_k, Hk, d] (the packed row layout);
 *       vt8 [Hk, d, kp] with kp = 16 * ceil(total_k / 16) + 16 * B: sequence b
 *       owns columns [c(b), c(b + 1)), c(b) = 16 * ceil(cu_k[b] / 16) + 16 * b,
 *       its keys in order and zeros after them.
 * fa_fp8_varlen_sizes    -- sizes[0..5] as fa_fp8_sizes, for these layouts.
 * fa_quantize_fp8_varlen -- fills them from packed bf16 q [total_q, H, d] and
 *                           k, v [total_k, Hk, d]; pointer rules as
 *                           fa_quantize_fp8.
 * fa_fwd_fp8_varlen      -- the forward on them: o bf16 [total_q, H, d], lse
 *                           fp32 [B, H, max_seqlen_q] (entries past a sequence's
 *                           length not written), flags 0 or FA_FLAG_CAUSAL
 *                           (bottom-right within each sequence); a sequence with
 *                           no keys gets o = 0 and lse = -inf.  Every pointer
 *                           non-NULL; d = 128 only.
 */
int fa_fp8_varlen_sizes(int B, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H, int Hk,
                        int d, long long* sizes);
int fa_quantize_fp8_varlen(const void* q, const void* k, const void* v, const int* cu_seqlens_q,
                           const int* cu_seqlens_k, int B, int total_q, int total_k, int max_seqlen_q,
                           int max_seqlen_k, int H, int Hk, int d, void* q8, void* k8, void* vt8, float* q_scale,
                           float* k_scale, float* v_scale, void* stream);
int fa_fwd_fp8_varlen(const void* q8, const void* k8, const void* vt8, const float* q_scale, const float* k_scale,
                      const float* v_scale, void* o, float* lse, const int* cu_seqlens_q, const int* cu_seqlens_k,
                      int B, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H, int Hk, int d,
                      float scale, int flags, void* stream);

/*
 * fa_set_timeout_ns -- limit for every device-side wait (mbarrier waits) in
 * later launches.  On expiry the kernel records FA_ERR_TIMEOUT, drains its
 * own copies and MMAs, releases tensor memory and exits.  Default 1e9 ns.
 * ns == 0 restores the default.
 */
int fa_set_timeout_ns(unsigned long long ns);

/*
 * Kernel configuration ("Flash Attention 2 Chapter6", Kernel 7: the
 * configuration space is searched per shape instead of fixed).  A config is
 * a text spec of comma-separated key=value items, any subset of
 *   br=<128|256>      query rows per work unit (B_r: one or two 128-row tiles)
 *   bc=<64|128>       keys per K/V tile (B_c)
 *   stages=<2|3|4>    slots of the shared-memory K/V ring (each holds one K
 *                     and one V tile; d = 128 with bc = 128 always uses 2,
 *                     the most that fit)
 *   threshold=<float> O-rescale threshold in log2 units, 0..64 (0 rescales
 *                     whenever a row maximum grows)
 * Items left out take br=256, bc=128, stages=4, threshold=8.  Causal calls
 * always use bc=128.  fa_get_config reports all four items as
 * "br=..,bc=..,stages=..,threshold=..".
 *
 * fa_set_config  -- force `spec` for every later call (NULL or "" clears it).
 * fa_get_config  -- writes the spec that a call with (d, N, varlen) would use
 *                   into buf (NUL-terminated, truncated to len); returns FA_OK.
 * fa_autotune    -- times every candidate config on the caller's tensors (same
 *                   arguments as fa_fwd), keeps the fastest for the key
 *                   (d, N bucket, varlen) and leaves the outputs written by
 *                   the winner.  Synchronises `stream`.
 */
int fa_set_config(const char* spec);
int fa_get_config(int d, int N, int varlen, char* buf, int len);
int fa_autotune(const void* q, const void* k, const void* v, void* o, float* lse, int B, int N,
                int H, int d, float scale, const int* cu_seqlens, void* stream);

/*
 * fa_selftest_wait_timeout -- launches one small kernel whose only work is an
 * mbarrier wait that nothing completes, bounded by `timeout_ns` (> 0, at most
 * 10 s).  It exercises the same bounded-wait routine as the attention kernel;
 * the expected outcome is FA_ERR_TIMEOUT from fa_check_status() with the
 * device still usable.  Returns FA_OK when the launch was enqueued.
 */
int fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

/*
 * fa_set_phase_buffer -- phase clocks for profiling the forward kernel's
 * pipeline (where each role of a CTA waits and works: "GPU 内核与 FlashAttention"
 * §8 asks where a kernel's time goes before tuning it).  Only the library
 * built with FA_PHASE_CLOCKS=1 (libfa_gb300_phase.so, `build.py --phase`)
 * records them; the default library returns FA_ERR_UNSUPPORTED and its
 * kernels contain none of the instrumentation.
 *   buf   : caller-owned DEVICE buffer of unsigned 64-bit words, 8-byte aligned,
 *           or NULL to detach.  Every forward launch that follows (bf16, key
 *           split, FP8) writes, for each CTA c, words [c * W, (c + 1) * W)
 *           with W the value returned: cycle counts per role (MMA issue,
 *           loads, the two softmax tiles, the epilogue) and the %globaltimer
 *           of the CTA's start and end.  The slot map is the PhaseBase /
 *           PhaseSlot enumeration of the kernel source.
 *   words : size of buf in words; a launch whose grid needs more returns
 *           FA_ERR_INVALID_ARG and launches nothing.  Work items: B * H *
 *           ceil(Nq / 256) for the dense forward, half as many when causal,
 *           times the splits for the key split.  Dense problems launch
 *           min(items, SMs) CTAs, packed batches one CTA per item, so items
 *           x W words always suffice; only the CTAs that run write their
 *           words (a CTA that takes over another's items leaves that CTA's
 *           words untouched).  When the
 *           buffer holds at least 3840 more words (3 units x 40 steps x 32
 *           events), an event trace follows the per-CTA words: clock64 stamps
 *           of each barrier hand-off of the first three work units of CTA 0
 *           (TraceEvent enumeration of the kernel source).
 * Returns W (> 0) on success, FA_ERR_INVALID_ARG for a too small or misaligned
 * buffer, FA_ERR_UNSUPPORTED in the default library.  Process-wide setting,
 * not thread-safe with respect to forward calls.
 */
int fa_set_phase_buffer(unsigned long long* buf, long long words);

/* Library version, major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_H */
