/*
 * xs.h - C ABI of libxs: non-causal attention fused with the post-attention
 * Ulysses All-to-All layout, for one GB300 (sm_103a).
 *
 * Source of the operations: "X-Stage: An Overlooked Pipeline Stage for
 * Communication-Computation Overlap in DiT Inference" (arXiv 2607.23264).
 *  - Abstract: for Ulysses sequence-parallel attention, the post-attention
 *    All-to-All is fused tile by tile into FlashAttention, so that the owner of
 *    an output tile issues its stores itself and resumes computation, with no
 *    dedicated communication warp or SM; compared against serial execution
 *    (FlashAttention, then the All-to-All) and FlashAttention alone.
 *  - Figure 5 (d)-(e): FlashAttention produces each head partition's output and
 *    the post-attention All-to-All restores the original sequence partition.
 *  - Figure 1 / Figure 7: the stores of one output tile drain while the next
 *    mainloop computes (the piggybacked FlashAttention-A2A pipeline).
 *
 * What every attention entry point computes, per batch b and head h:
 *     o[b][h][n][:] = softmax_j( q[b][h][n][:] . k[b][h][j][:] / sqrt(d) ) v[b][h][j][:]
 * over all N keys (non-causal, no mask, no dropout), fp32 accumulation, output
 * rounded to bf16 (round to nearest even).
 *
 * The layout ("shards"): destination p (0 <= p < P) receives the contiguous
 * sequence block [p*N/P, (p+1)*N/P) of every head:
 *     shard_p[b][i][h][c] = o[b][h][p*(N/P) + i][c],   0 <= i < N/P.
 * On one GPU the P destinations are P separate device buffers.
 *
 * Conventions shared by all calls
 *  - Element type: every buffer is bf16 (2 bytes), in device memory.
 *  - q, k, v, o: [B][H][N][d], contiguous (d fastest).
 *  - shard p: [B][N/P][H][d], contiguous; out_shards is a HOST array of P
 *    device pointers, read during the call (the array may be freed afterwards).
 *  - Ownership: the caller owns every buffer. The library allocates no device
 *    memory; it keeps only a device status word (see xs_last_device_status)
 *    and the fixed scratch array of xs_attn_serial_noalloc. An optional
 *    caller-owned workspace (xs_set_workspace) enables a balanced schedule.
 *  - Asynchrony: each call only enqueues work on `stream` (a cudaStream_t; NULL
 *    means the legacy default stream) and returns without synchronising. Launch
 *    errors are reported as XS_ERR_CUDA. Kernel-side waits are bounded: a wait
 *    that runs out records XS_ERR_TIMEOUT in the status word and the kernel
 *    returns, leaving the context usable.
 *  - Aliasing: inputs, outputs and shards must not overlap.
 *  - Threads: calls on different streams are independent.
 *  - Validation, in this order, before any device work:
 *      XS_ERR_INVALID     a NULL pointer (also any NULL shard), B, N or H < 0,
 *                         P not in [1, 8], N % P != 0,
 *                         store_tile not in {1, 2, 4, 8};
 *      XS_ERR_UNSUPPORTED d not in {64, 128, 256}, N % 128 != 0, d = 256
 *                         with store_tile != 8 (at d = 256 every finished tile
 *                         is stored at once: a deferred tile does not fit on
 *                         chip beside the K/V ring), or B*H*N >= 2^31 (the
 *                         kernels address rows with 32-bit coordinates);
 *      XS_ERR_ALIGN       a pointer that is not 16-byte aligned.
 *    B == 0, H == 0 or N == 0 is an empty problem: the call validates its
 *    other arguments and returns XS_OK without launching anything.
 */
#ifndef XS_H
#define XS_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  XS_OK = 0,
  XS_ERR_INVALID = 1,
  XS_ERR_UNSUPPORTED = 2,
  XS_ERR_ALIGN = 3,
  XS_ERR_CUDA = 4,
  XS_ERR_TIMEOUT = 5
} xs_status;

/* Fused attention + shard layout (abstract: tile-granular fusion of the
 * post-attention All-to-All with FlashAttention; Figure 7). One persistent
 * kernel (d = 64 and 128: two query tiles per CTA; d = 256: one query tile per
 * CTA with its scores double-buffered on chip). Each finished 128-row output
 * tile is staged on chip and written into the P shards by the warps that own
 * it, in bursts of `store_tile` 16-row slabs interleaved with the KV
 * iterations of that warp group's next tile (store_tile = 8, or a tile with no
 * next tile on its SM: the whole tile right after it is finished).
 * The result does not depend on store_tile.
 *   q, k, v     [B][H][N][d] bf16, device.
 *   out_shards  host array of P device pointers, shard p [B][N/P][H][d] bf16.
 *   store_tile  1, 2, 4 or 8 slabs per burst (8 only at d = 256). */
xs_status xs_attn_fused(const void *q, const void *k, const void *v,
                        void *const *out_shards, int B, int N, int H, int d,
                        int P, int store_tile, void *stream);

/* Flags of xs_attn_fused_ex. */
#define XS_FLAG_COMPLETION_COUPLED 1

/* xs_attn_fused with two experiment controls for the residual-slope test
 * (Pith review of X-Stage, "If this is right": the completion-coupled model,
 * where the issuer is blocked until its stores are visible, predicts a
 * residual over FlashAttention alone that grows linearly with sequence length,
 * while X-Stage predicts a flat one; Figure 11 caption: relative
 * sender-visible residual E_res(M)/T_FA; referee summary: per-tile
 * remote-store span distributions).
 *   flags  0, or XS_FLAG_COMPLETION_COUPLED: after issuing a finished tile's
 *          stores the issuing thread waits until they have completed before
 *          its warp group resumes (requires store_tile 8).
 *   spans  NULL, or a device buffer of 2*B*H*(N/128) unsigned 64-bit values,
 *          all zero on entry (8-byte aligned): for output tile
 *          t = (b*H + h)*(N/128) + n/128, spans[2t] and spans[2t + 1] receive
 *          the %globaltimer (ns) at which its first slab was issued and at which
 *          the last of its issuing warps was released.
 * Output bytes are identical to xs_attn_fused. Other flag bits, or the
 * coupled flag with store_tile != 8: XS_ERR_INVALID. */
xs_status xs_attn_fused_ex(const void *q, const void *k, const void *v,
                           void *const *out_shards, int B, int N, int H, int d,
                           int P, int store_tile, int flags,
                           unsigned long long *spans, void *stream);

/* Attention alone (the FlashAttention-alone time the abstract compares the
 * fused kernel with): same kernel, output written head-major to
 * o [B][H][N][d] bf16 (device). */
xs_status xs_attn(const void *q, const void *k, const void *v, void *o, int B,
                  int N, int H, int d, void *stream);

/* The layout alone (the separate post-attention All-to-All of serial
 * execution, Figure 5 (e)), as a bit-exact copy kernel:
 * o [B][H][N][d] -> shards. Any 16-bit payload is copied unchanged. */
xs_status xs_scatter(const void *o, void *const *out_shards, int B, int N,
                     int H, int d, int P, void *stream);

/* Serial execution (abstract: the baseline of the sender-visible speedup):
 * xs_attn into the caller's o_scratch [B][H][N][d] bf16, then xs_scatter into
 * the shards, two launches on `stream`. o_scratch holds o afterwards. */
xs_status xs_attn_serial(const void *q, const void *k, const void *v,
                         void *o_scratch, void *const *out_shards, int B, int N,
                         int H, int d, int P, void *stream);

/* Ulysses sequence-parallel attention with BOTH All-to-Alls fused (Figure 5:
 * QKV projection and the pre-attention All-to-All turn sequence-partitioned
 * tokens into head partitions (a)-(c); FlashAttention and the post-attention
 * All-to-All produce the output and restore the sequence partition (d)-(e)).
 * The inputs stay in the sequence partition: q_shards[p], k_shards[p],
 * v_shards[p] (host arrays of P device pointers) are [B][N/P][H_total][d] bf16,
 * the tokens [p*N/P, (p+1)*N/P) of every head, as each rank holds them after
 * the QKV projection. The call computes attention over all N tokens for the
 * heads [h0, h0 + H) only (the head partition one rank owns after the
 * pre-attention All-to-All), reading its Q/K/V tiles straight from the
 * sequence shards, and stores output row n of head h0 + h into
 * out_shards[n / (N/P)][b][n % (N/P)][h0 + h][:] (destinations [B][N/P][H_total][d]),
 * the owner of each tile issuing the stores as in xs_attn_fused. On one GPU,
 * h0 = 0 and H = H_total does the whole layer; P calls with
 * h0 = r*H_total/P, H = H_total/P do rank r's share each.
 * Validation as xs_attn_fused, plus: XS_ERR_INVALID for NULL arrays or
 * entries, H_total < 1, h0 < 0, H < 0 or h0 + H > H_total;
 * XS_ERR_UNSUPPORTED unless N/P is a multiple of 128 (a 128-row tile never
 * straddles two input shards); XS_ERR_ALIGN for unaligned shard pointers.
 * H == 0 is an empty call. Heads outside [h0, h0 + H) of the destinations are
 * not touched. */
xs_status xs_attn_ulysses(const void *const *q_shards, const void *const *k_shards,
                          const void *const *v_shards, void *const *out_shards, int B,
                          int N, int H_total, int h0, int H, int d, int P,
                          int store_tile, void *stream);

/* Store-burst probe for the Burst-Gap model (Pith review of X-Stage, "What
 * carries the argument" and "What would settle it": zero-gap periodic bursts
 * give the drain rate R, a recovered large-gap plateau the backpressure-free
 * issue time T_iss^0, the isolated-burst knee the outstanding capacity Q;
 * Figure 3 caption). Local form: the stores go to this GPU's own memory.
 * K producer CTAs (128 threads each) each issue n_bursts bursts of burst_bytes
 * into fresh memory, separated by gap_ns nanoseconds without stores. For
 * producer c and burst b, times[2*(c*n_bursts + b)] and [.. + 1] receive the
 * %globaltimer values (ns) at which the CTA started issuing the burst and at
 * which every store had been issued.
 *   dst       device buffer of dst_bytes >= K*n_bursts*burst_bytes (16-byte aligned)
 *   times     device buffer of 2*K*n_bursts unsigned 64-bit values (8-byte aligned)
 *   mode      0: posted st.global.v4 from all threads; 1: TMA bulk copies from
 *             shared memory, span ending when their source has been read
 *   XS_ERR_INVALID for NULL pointers, K not in [1, 1024], n_bursts < 1,
 *   burst_bytes not a positive multiple of 2048, gap_ns > 1e9, a bad mode or a
 *   too small dst; XS_ERR_ALIGN for misaligned pointers. */
xs_status xs_store_burst_probe(void *dst, unsigned long long dst_bytes, int K,
                               unsigned long long burst_bytes, int n_bursts,
                               unsigned long long gap_ns, int mode,
                               unsigned long long *times, void *stream);

/* Size of the scratch array that xs_attn_serial_noalloc uses: 32 MiB. */
#define XS_NOALLOC_SCRATCH_BYTES (32ull << 20)

/* Serial execution without a caller-supplied intermediate buffer, for callers
 * that cannot allocate device memory (for example code embedded in a host
 * framework that owns all device memory through its own allocator or a fixed
 * memory plan, or loops where a cudaMalloc would synchronise the device).
 * The paper has no counterpart to this entry point; it only changes where the
 * intermediate o of xs_attn_serial lives.
 * Same arguments, results and validation as xs_attn_serial minus o_scratch:
 * the intermediate o [B][H][N][d] bf16 lives in one array of
 * XS_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that
 * loads the library holds until the process exits. Nothing is allocated:
 * no cudaMalloc, cudaFree or allocating library call.
 *   - XS_ERR_INVALID if B*H*N*d*2 bytes exceed XS_NOALLOC_SCRATCH_BYTES
 *     (checked first, factor by factor so no product wraps, before any device
 *     work).
 *   - Every call looks up the array's device address on the current device
 *     (a symbol lookup, no allocation), so a device reset that reloads the
 *     library's device code cannot leave a stale address in use. The first
 *     call on a device may load that code: make it before any stream capture.
 *   - Every call on a device shares the one array and leaves the last call's o
 *     in it (each call overwrites all of the o it reads, so nothing needs
 *     clearing). Calls that overlap on the GPU (different streams, or
 *     different host threads without ordering) race on the array. */
xs_status xs_attn_serial_noalloc(const void *q, const void *k, const void *v,
                                 void *const *out_shards, int B, int N, int H,
                                 int d, int P, void *stream);

/* Balanced schedule with a workspace (a scheduling aid of this implementation;
 * the paper has no counterpart). The attention kernel runs one persistent CTA
 * per SM. Without a workspace each CTA takes whole units (a head and a pair of
 * 128-row query tiles) in turn, so when the units do not divide evenly over
 * the SMs the last wave leaves SMs idle. With a workspace the launch may
 * instead give every CTA an equal contiguous range of the (unit, 128-key tile)
 * iterations (a "stream-K" schedule): a unit cut by a range boundary is
 * computed in pieces on consecutive CTAs, each piece leaves its partial result
 * (unnormalised output rows, running maximum, row sum; fp32) in the workspace,
 * and the CTA finishing a unit's last piece merges the pieces with the
 * online-softmax rescaling identity and stores the output tile as usual (into
 * o, or into the shards). The library chooses per launch, from the shape and
 * the SM count, whichever schedule its cost model finds shorter. Results agree
 * with the whole-unit schedule within fp32 rounding of the merge (they are not
 * bit-identical to it) and are identical from launch to launch.
 *
 * XS_WORKSPACE_HEADER_BYTES: the first bytes of a workspace hold per-unit
 * counters that must be zero before a launch; the launches leave them zero. */
#define XS_WORKSPACE_HEADER_BYTES 16384ull

/* Registers (ws != NULL) or removes (ws == NULL) the caller's device workspace
 * for the current device. Later attention launches on that device (every entry
 * point above that computes attention) use it when the balanced schedule is
 * shorter and `bytes` suffice; otherwise they take whole units. The caller
 * keeps ownership and must keep the buffer alive until it removes it.
 *   ws     device memory, 256-byte aligned (XS_ERR_ALIGN otherwise)
 *   bytes  >= XS_WORKSPACE_HEADER_BYTES (XS_ERR_INVALID otherwise)
 * The call zeroes the header on `stream` and synchronises it (XS_ERR_CUDA on
 * failure). Launches that use one workspace must not overlap on the GPU
 * (different streams without ordering race on it). After a launch reported
 * XS_ERR_TIMEOUT (xs_last_device_status), register the workspace again to
 * re-zero its counters. */
xs_status xs_set_workspace(void *ws, unsigned long long bytes, void *stream);

/* For an attention launch of this shape on the current device with an
 * unlimited workspace: *bytes = the workspace it would use and *cut = 1 if it
 * would take the balanced schedule (*bytes = 0 and *cut = 0 for whole units).
 * cut may be NULL. XS_ERR_INVALID for a NULL bytes or B, N, H < 0;
 * XS_ERR_UNSUPPORTED for d not in {64, 128, 256} or N % 128 != 0; XS_ERR_CUDA if
 * the device cannot be queried. */
xs_status xs_workspace_bytes(int B, int N, int H, int d, unsigned long long *bytes, int *cut);

/* Static English text for a status code; never NULL. */
const char *xs_status_string(xs_status s);

/* Synchronises `stream`, then reads and clears the library's device status
 * word for the current device: XS_ERR_TIMEOUT if a kernel's bounded wait ran
 * out since the last call, XS_ERR_CUDA if the synchronisation failed, else
 * XS_OK. For tests and debugging; the attention calls never block on it. */
xs_status xs_last_device_status(void *stream);

/* Sets the limit, in nanoseconds, after which a kernel's on-chip wait gives up
 * (default 2e9 = 2 s; 0 restores the default). Applies to later launches from
 * this process. Returns the previous limit. */
unsigned long long xs_set_wait_limit_ns(unsigned long long limit_ns);

/* Self-test of the bounded wait: launches one CTA that waits on an on-chip
 * barrier that nothing ever signals, with the current wait limit. The wait
 * must run out, record XS_ERR_TIMEOUT in the status word and return. Read the
 * outcome with xs_last_device_status. */
xs_status xs_selftest_bounded_wait(void *stream);

/* Self-test of the softmax's two exponential paths: for i < n (device fp32
 * buffers), out_poly[i] = 2^x[i] as the attention kernel's polynomial computes
 * it on the FMA pipe for a share of each row (range reduction x = n + f,
 * degree-3 minimax polynomial for 2^f, n added to the exponent; arguments below
 * -126 raised to -126), out_mufu[i] = 2^x[i] from the MUFU unit (ex2.approx,
 * subnormal results flushed to zero). For tests comparing the two against each
 * other and against an error bound. XS_ERR_INVALID for NULL pointers or n < 0. */
xs_status xs_selftest_exp2(const float *x, float *out_poly, float *out_mufu, int n, void *stream);

/* ABI version of this header (1). */
int xs_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* XS_H */
