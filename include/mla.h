/*
 * mla.h — C ABI of libmla: Multi-head Latent Attention (MLA) decode with
 * matrix absorption over a paged latent KV cache, for one NVIDIA GB300
 * (sm_103a).
 *
 * Method (cited by page and section):
 *   - MLA operator write-up (nxmr.cn/news/151634) §1: every cached token of a
 *     layer holds a 512-d latent c_KV plus a 64-d decoupled RoPE key k_R,
 *     576 elements, 1.125 KB in bf16.
 *   - same page §4 (the absorption-equivalence script): K = c_KV·W_UK^T per
 *     head ("path A") equals absorbing W_UK into the query,
 *     q_abs = q_nope·W_UK ("path B"); score = (q_abs·c_KV + q_R·k_R) · scale
 *     with scale = (d_hc + d_R)^-1/2 = 1/sqrt(192).
 *   - same page §3: page_size 64 (a 64-token page is 73,728 B and suits bulk
 *     tensor copies), tile of 64 tokens, multi-stage pipeline.
 *   - "From MLA to GLA" (hotelren.com/news/5324130) §1: grouped latent
 *     attention (GLA), heads split into groups that each own a latent.
 *
 * One decode step of one layer is four calls on one stream:
 *   mla_absorb_q  →  mla_decode_paged  →  mla_combine_splits  →  mla_project_uv
 * or three, with the last two fused:
 *   mla_absorb_q  →  mla_decode_paged  →  mla_combine_project
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers owned by the caller. The
 *     library never allocates device memory and never synchronises the
 *     stream except in mla_get_device_status.  Its only state is a
 *     per-device cache of launch limits (found on first use, guarded by a
 *     mutex), a cache of the 64 tensor maps encoded last (keyed by every
 *     encoding argument, the buffer address included; guarded by a mutex),
 *     and the scratch array of mla_decode_attend_noalloc.
 *   - bf16 tensors are passed as raw 16-bit storage (void*); fp32 as float*;
 *     indices as int32.  All tensors are dense, row-major, no padding.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *     is the legacy default stream).  The int return value reports argument
 *     validation and launch errors only (mla_status).  Errors found on the
 *     device (bad block_table entry, bad sequence length, a bounded wait that
 *     gave up) are written to a sticky status word inside the decode
 *     workspace; read it with mla_get_device_status.
 *   - Nothing is thrown across the ABI.  Every call is thread-safe as long as
 *     concurrent calls do not share output buffers or workspaces.
 *   - mla_absorb_q, mla_decode_paged and mla_project_uv launch their kernels
 *     with programmatic dependent launch: a kernel may start its on-chip
 *     set-up while the kernel before it on the stream is still running, but
 *     reads and writes global memory only after that kernel has completed.
 *     Stream order therefore holds for every caller kernel in between, as
 *     for ordinary launches.
 *
 * Notation (dims struct):
 *   B batch, Lq new tokens per sequence, H heads, d_hc = 128 content head dim,
 *   d_c = 512 latent width, d_R = 64 RoPE width, G latent groups (1 = MLA,
 *   2, 4 or 8 = GLA), d_g = d_c / G latent width per group, P = page_size =
 *   64.
 *   Head h belongs to group g(h) = floor(h * G / H) (contiguous head blocks).
 *   Cache row of one token = [c_0 | ... | c_{G-1} | k_R], d_c + d_R = 576 bf16.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mla_dims {
  int B;                 /* batch (sequences), >= 1                          */
  int Lq;                /* new query tokens per sequence, 1..4              */
  int H;                 /* heads, multiple of 16, 16..128                   */
  int d_hc;              /* content head dim, must be 128                    */
  int d_c;               /* total latent width, must be 512                  */
  int d_R;               /* decoupled RoPE width, must be 64                 */
  int G;                 /* latent groups: 1 (MLA), 2, 4 or 8 (GLA)          */
  int page_size;         /* tokens per cache page, must be 64                */
  int max_pages_per_seq; /* row length of block_table                        */
  int num_pages;         /* physical pages in the cache                      */
  float scale;           /* softmax scale, normally 1/sqrt(d_hc + d_R)       */
  int causal;            /* 1: query l sees keys 0 .. n-Lq+l (required if Lq>1) */
} mla_dims;

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,  /* null pointer, non-positive size, bad scale  */
  MLA_ERR_UNSUPPORTED = -2,  /* dims outside the supported set above       */
  MLA_ERR_MISALIGNED = -3,   /* a pointer is not 16-byte aligned           */
  MLA_ERR_WORKSPACE = -4,    /* workspace missing or too small             */
  MLA_ERR_CUDA = -5,         /* a CUDA runtime / driver call failed        */
  MLA_ERR_BAD_TABLE = -6,    /* device: block_table entry out of range     */
  MLA_ERR_BAD_SEQLEN = -8,   /* device: seq_len < Lq or > max_pages*P      */
  MLA_ERR_TIMEOUT = -7,      /* device: a bounded pipeline wait gave up    */
  MLA_ERR_RANGE = -9         /* device (FP8 cache): a scale or a query value
                                outside the range of the f16 arithmetic    */
} mla_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* mla_status_string(int status);

/*
 * mla_absorb_q — absorb W_UK into the query (MLA operator write-up §4,
 * "path B": einsum qhd,hdc->qhc) and append the RoPE part.
 *
 *   q_cat[b,l,h, 0:d_g]        = bf16( sum_d q_nope[b,l,h,d] * W_UK[h,d,:] )
 *   q_cat[b,l,h, d_g:d_g+d_R]  = q_rope[b,l,h,:]
 *
 * q_nope bf16 [B,Lq,H,d_hc]; q_rope bf16 [B,Lq,H,d_R];
 * W_UK bf16 [H,d_hc,d_g] (head h's block maps the 128-d content query to its
 * group's d_g-wide latent); q_cat bf16 [B,Lq,H,d_g+d_R] (output).
 * fp32 accumulation on the tensor cores, one rounding to bf16.
 * Errors: MLA_ERR_INVALID_ARG (null), MLA_ERR_UNSUPPORTED (dims),
 * MLA_ERR_MISALIGNED (any pointer not 16-byte aligned), MLA_ERR_CUDA.
 */
int mla_absorb_q(const mla_dims* dims, const void* q_nope, const void* q_rope,
                 const void* W_UK, void* q_cat, void* stream);

/*
 * Number of partial-output slots mla_decode_paged writes for these dims on
 * the current device (depends on the device's SM count).  o_part must hold
 * slots * Lq*H * d_c floats and lse_part slots * Lq*H floats.
 */
int mla_decode_num_slots(const mla_dims* dims, int* slots);

/*
 * Number of kernels one mla_decode_paged call with these dims launches: 1
 * when B <= 448 for G = 1, B <= 352 for G > 1 (the decode kernel computes
 * its own split of the work, one sequence per thread), 2 above that (a plan
 * kernel runs first).  Host-only, launches nothing.
 */
int mla_decode_kernel_launches(const mla_dims* dims, int* launches);

/*
 * Bytes of workspace mla_decode_paged needs (split plan + sticky status
 * word).  The caller allocates it, zero-fills it ONCE (that clears the status
 * word) and may reuse it for any number of calls with the same or smaller
 * dims.
 */
int mla_decode_workspace_size(const mla_dims* dims, size_t* bytes);

/*
 * mla_decode_paged — split-KV flash-decoding over the paged latent cache.
 *
 * Source: the attention of the MLA operator write-up §4 ("path B": scores
 * from the absorbed query against the cached latent and RoPE key, scale
 * (d_hc + d_R)^-1/2) over the paged cache of §1/§3 (row = 512-d latent +
 * 64-d RoPE key, 64-token pages).  The split into key ranges with a
 * per-range (o, lse) and the causal window of multi-token decode are not on
 * the pages (they are silent on both); the split is flash-decoding's, and
 * the window is the plainest reading: query l of Lq new tokens sees every
 * key up to and including its own position.
 *
 * For each sequence b (n = seq_lens[b] cached tokens, the last Lq of them
 * being the new tokens) and query row (l, h) with visible keys
 * s = 0 .. n-Lq+l:
 *     score_s = (q_cat[b,l,h,0:d_g] . c_{g(h)}[s] + q_cat[b,l,h,d_g:] . k_R[s]) * scale
 * over the cache rows gathered through block_table (token s of sequence b is
 * row s % P of physical page block_table[b, s / P]).  The work is split into
 * contiguous page ranges; each range produces, per query row, the normalised
 * latent partial o = sum_s p_s c_{g(h)}[s] / sum_s p_s and its natural-log
 * log-sum-exp lse = log sum_s exp(score_s) (-inf for an empty range).
 *
 * q_cat    bf16 [B,Lq,H,d_g+d_R] (from mla_absorb_q), 16-byte aligned
 * kv_cache bf16 [num_pages, P, d_c+d_R], 16-byte aligned.  Whole pages are
 *          read: the rows of a sequence's last page past its end take part
 *          in the tensor-core products with weight 0, so they must hold
 *          finite values of the cache's usual size (zeros, or rows left
 *          from earlier sequences); a NaN there would reach the output
 *          (0 * NaN), a huge value would coarsen the partial scores' 16-bit
 *          scale.  (The decompress branch has no such condition.)
 * block_table int32 [B, max_pages_per_seq]; entries past ceil(n/P) unused
 * seq_lens int32 [B]
 * o_part  fp32 scratch of slots * Lq*H * d_c floats for mla_combine_splits
 *         (its layout is private to the library), 16-byte aligned
 * lse_part fp32 [slots, Lq*H]
 * workspace / ws_bytes: see mla_decode_workspace_size.
 * num_splits: 0 = automatic (all SMs busy); otherwise the number of
 *   concurrent work units (CTA clusters) to use, clamped to the device.
 * Errors: synchronous MLA_ERR_INVALID_ARG / UNSUPPORTED / MISALIGNED /
 * WORKSPACE / CUDA; asynchronous MLA_ERR_BAD_TABLE, MLA_ERR_BAD_SEQLEN,
 * MLA_ERR_TIMEOUT into the workspace status word.  Out-of-range table
 * entries are never dereferenced (clamped, and the status is set).
 */
int mla_decode_paged(const mla_dims* dims, const void* q_cat,
                     const void* kv_cache, const int32_t* block_table,
                     const int32_t* seq_lens, int num_splits, float* o_part,
                     float* lse_part, void* workspace, size_t ws_bytes,
                     void* stream);

/*
 * mla_decode_paged_fp8 — mla_decode_paged over a latent cache stored in FP8
 * with the latent dequantised on load.
 *
 * Source: the MLA operator write-up (nxmr.cn/news/151634), introduction and
 * the tail of §5: a low-precision (NVFP4) KV cache read with 16-byte vector
 * loads from 16-byte aligned pages.  The pages fix neither the format nor
 * the scales; this entry takes the plainest FP8 reading: OCP e4m3 codes
 * (bias 7, no infinities, 0x7f/0xff NaN) with one power-of-two scale per
 * token and 128-column block of the latent; the RoPE key stays bf16.
 *
 * kv_cache_fp8: [num_pages, P, 656] bytes, 16-byte aligned; row of a token:
 *   bytes   0..511  e4m3 codes of c_KV (group g's latent is codes
 *                   g*d_g .. (g+1)*d_g - 1)
 *   bytes 512..639  k_R, 64 bf16
 *   bytes 640..655  4 fp32 scales; scale j applies to codes 128j..128j+127
 * The latent the attention sees is c[i] = e4m3(code[i]) * scale[i / 128];
 * everything else (arguments, outputs, split, errors) is as for
 * mla_decode_paged, whose o_part, lse_part and workspace this call fills in
 * the same form (merge them with mla_combine_splits or mla_combine_project).
 *
 * The latent products run on f16 tensor-core operands: the dequantised
 * value is exact in f16 when the scale is 0 or a power of two in
 * [2^-15, 2^7] (another value in that range is rounded to f16 once); the
 * query's latent part (q_cat[..., 0:d_g], bf16) is converted to f16, exact
 * within +-65504; the softmax weights are rounded to f16 (bf16 in
 * mla_decode_paged).  A scale that is neither 0 nor in that range, on any
 * row of a page the call reads (rows past a sequence's end included: they
 * enter the products with weight 0, and an infinite value would turn that
 * into NaN), or a query value beyond 65504, sets MLA_ERR_RANGE in the status
 * word.  Codes past a sequence's end must not be NaN (0x7f, 0xff); zero
 * filled rows are fine.
 */
int mla_decode_paged_fp8(const mla_dims* dims, const void* q_cat,
                         const void* kv_cache_fp8, const int32_t* block_table,
                         const int32_t* seq_lens, int num_splits, float* o_part,
                         float* lse_part, void* workspace, size_t ws_bytes,
                         void* stream);

/*
 * mla_combine_splits — merge the split partials of mla_decode_paged by
 * log-sum-exp (flash-decoding reduction; the pages are silent on the merge,
 * this is the exact identity of a softmax taken over disjoint key ranges):
 *     L = log sum_k exp(lse_k),   o_lat = sum_k exp(lse_k - L) * o_k
 * Ranges with lse = -inf contribute nothing.
 * o_part / lse_part / workspace: exactly as passed to mla_decode_paged (the
 * workspace carries the split plan).  o_lat bf16 [B,Lq,H,d_g] (each head's
 * own group slice of the latent); lse fp32 [B,Lq,H] (may be NULL).
 */
int mla_combine_splits(const mla_dims* dims, const float* o_part,
                       const float* lse_part, const void* workspace,
                       size_t ws_bytes, void* o_lat, float* lse, void* stream);

/*
 * mla_project_uv — map the latent output back to the head dimension with
 * W_UV (the up-projection of the values, applied after attention; the MLA
 * operator write-up §1 says only that the latent is mapped back to the high
 * dimension when needed, the absorbed form of V = c . W_UV^T per head):
 *     out[b,l,h,:] = W_UV[h] (d_hc x d_g) . o_lat[b,l,h,:]
 * o_lat bf16 [B,Lq,H,d_g]; W_UV bf16 [H,d_hc,d_g]; out bf16 [B,Lq,H,d_hc].
 * fp32 accumulation on the tensor cores.
 */
int mla_project_uv(const mla_dims* dims, const void* o_lat, const void* W_UV,
                   void* out, void* stream);

/*
 * Testing hook for the decode kernel's timeout path (no counterpart in the
 * source pages), process-wide, for the mla_decode_paged launches that
 * follow:
 *   wait_limit_ns  wall-clock limit of every wait between the kernel's warps
 *                  (0 restores the default, 2 s);
 *   stall_page     >= 0: before the QK of that page of its work unit, each
 *                  CTA's MMA-issuing thread also waits on a barrier that
 *                  nothing completes, so that wait gives up after the limit
 *                  (-1 restores the default: no such wait).
 * A wait that gives up records MLA_ERR_TIMEOUT in the workspace status word;
 * the kernel then waits for the copies and MMAs it started and returns.
 * Nothing is skipped and no memory is touched out of bounds, so the context
 * stays usable.  Errors: MLA_ERR_INVALID_ARG (wait_limit_ns < 0 or
 * stall_page < -1).
 */
int mla_set_timeout_test(long long wait_limit_ns, int stall_page);

/*
 * mla_combine_project — mla_combine_splits and mla_project_uv in one kernel:
 * the merged latent rows of each head go straight into on-chip memory as
 * the operand of the W_UV product, so o_lat never makes a round trip
 * through device memory (the MLA operator write-up §1 points out that
 * intermediate reads and writes eat the absorbed path's gains).
 *     out[b,l,h,:] = W_UV[h] . sum_k exp(lse_k - L) o_k,   L = log sum_k exp(lse_k)
 * o_part / lse_part / workspace: as passed to mla_decode_paged.  W_UV and
 * out: as for mla_project_uv.  o_lat (bf16 [B,Lq,H,d_g]) and lse (fp32
 * [B,Lq,H]) are also written when not NULL.  Same rounding as the two calls
 * (o_lat rounded to bf16 before the product).
 * Errors: MLA_ERR_INVALID_ARG / UNSUPPORTED / MISALIGNED / WORKSPACE / CUDA.
 */
int mla_combine_project(const mla_dims* dims, const float* o_part,
                        const float* lse_part, const void* workspace,
                        size_t ws_bytes, const void* W_UV, void* out,
                        void* o_lat, float* lse, void* stream);

/*
 * mla_decode_step — one whole decode step in one call, for callers that
 * would otherwise pay a host round trip per call:
 *     mla_absorb_q -> mla_decode_paged (kv_fp8 = 0) or mla_decode_paged_fp8
 *     (kv_fp8 != 0) with automatic splits -> mla_combine_splits +
 *     mla_project_uv (fused = 0) or mla_combine_project (fused != 0)
 * on `stream`, with the arguments, buffers and errors of those calls (the
 * first error is returned and nothing after it is launched).  o_lat is
 * required unless fused; lse may be NULL.  The same kernels as the separate
 * calls, so the results are identical.
 */
int mla_decode_step(const mla_dims* dims, const void* q_nope, const void* q_rope,
                    const void* W_UK, const void* W_UV, const void* kv_cache,
                    int kv_fp8, const int32_t* block_table,
                    const int32_t* seq_lens, void* q_cat, float* o_part,
                    float* lse_part, void* workspace, size_t ws_bytes,
                    void* o_lat, float* lse, void* out, int fused,
                    void* stream);

/*
 * ---- The decompress branch, for long query chunks.
 * The MLA operator write-up §3 (the plugin's prefill threshold of 256 query
 * tokens) and §6 (long chunks decompress K and V and run ordinary attention;
 * short ones stay in the latent space): callers with Lq >= the threshold
 * take mla_decompress_kv + mla_prefill_attend; mla_decode_paged serves
 * Lq <= 4.  Both calls accept any 1 <= Lq <= max_pages_per_seq * 64; the
 * other dims are as for the decode (G in {1, 2, 4, 8}).
 */
#define MLA_PREFILL_THRESHOLD 256

/*
 * Bytes of ONE of the two buffers mla_decompress_kv writes (k_nope or v):
 * B * H * max_pages_per_seq * 64 * d_hc bf16 values.
 */
int mla_decompressed_kv_size(const mla_dims* dims, size_t* bytes);

/*
 * mla_decompress_kv — per-head keys and values from the latent cache (the
 * write-up's §1: MLA stores c and recovers K and V by the up-projections;
 * §4: K = c . W_UK^T, the same orientation as the absorption):
 *     k_nope[b,h,s,:] = W_UK[h] . c_g(h)[s],   v[b,h,s,:] = W_UV[h] . c_g(h)[s]
 * for every cached token s < seq_lens[b] (read through block_table as in
 * mla_decode_paged), and zeros for the rest of the sequence's last page.
 * k_nope, v: bf16 [B, H, max_pages_per_seq * 64, d_hc], caller-allocated
 * (mla_decompressed_kv_size bytes each); rows past the last page are not
 * written.  workspace: at least 32 bytes whose first int is the sticky
 * status word (a decode workspace will do), zeroed once by the caller; bad
 * table entries (MLA_ERR_BAD_TABLE) and lengths (MLA_ERR_BAD_SEQLEN: outside
 * [Lq, max_pages_per_seq * 64]) are recorded there and clamped, never
 * dereferenced.  fp32 accumulation on the tensor cores, bf16 out.
 * Errors: MLA_ERR_INVALID_ARG / UNSUPPORTED / MISALIGNED (16 bytes for the
 * tensors, 4 for the index arrays and workspace) / WORKSPACE / CUDA.
 */
int mla_decompress_kv(const mla_dims* dims, const void* kv_cache,
                      const int32_t* block_table, const int32_t* seq_lens,
                      const void* W_UK, const void* W_UV, void* k_nope, void* v,
                      void* workspace, size_t ws_bytes, void* stream);

/*
 * mla_prefill_attend — causal attention of Lq new tokens over the
 * decompressed keys and values (the write-up's §4 "path A", the
 * non-absorbed form):
 *     out[b,l,h,:] = sum_s p_s v[b,h,s,:],
 *     p = softmax_s((q_nope[b,l,h] . k_nope[b,h,s] + q_rope[b,l,h] . k_R[s]) * scale)
 * over the keys s <= seq_lens[b] - Lq + l (the new tokens are the last Lq of
 * the sequence), k_R[s] read from the cache row (columns 512..575).  lse
 * (fp32 [B,Lq,H]) receives the natural log-sum-exp of the scaled scores.
 * q_nope bf16 [B,Lq,H,d_hc], q_rope bf16 [B,Lq,H,d_R]; k_nope, v as written
 * by mla_decompress_kv; out bf16 [B,Lq,H,d_hc]; workspace, block_table,
 * seq_lens and errors as for mla_decompress_kv.  fp32 scores, fp32 online
 * softmax, bf16 weights P, fp32 accumulation.
 */
int mla_prefill_attend(const mla_dims* dims, const void* q_nope, const void* q_rope,
                       const void* kv_cache, const int32_t* block_table,
                       const int32_t* seq_lens, const void* k_nope, const void* v,
                       void* out, float* lse, void* workspace, size_t ws_bytes,
                       void* stream);

/*
 * Synchronise `stream`, then return the sticky device status of `workspace`
 * (MLA_OK or the first device error recorded since the workspace was zeroed).
 */
int mla_get_device_status(const void* workspace, void* stream);

/*
 * mla_decode_attend_noalloc — mla_decode_paged followed by
 * mla_combine_splits, for callers that cannot allocate device memory.
 * This is a library convenience with no counterpart in the source pages.
 *
 * Who it is for: callers that cannot hand the library scratch memory, e.g.
 * an engine whose memory planner has already given out all of the GPU, a
 * plugin inside a host program that owns every allocation, or a decode loop
 * recorded into a CUDA graph (where a cudaMalloc would break the capture).
 * They pass only inputs and outputs; the split plan, the status word and the
 * split partials live in one fixed 32 MiB array that the library reserves on
 * every GPU where it is loaded, until the process exits.
 *
 * q_cat, kv_cache, block_table, seq_lens: as for mla_decode_paged.
 * o_lat bf16 [B,Lq,H,d_g], lse fp32 [B,Lq,H] (may be NULL): as for
 * mla_combine_splits.  device_status (device int, may be NULL): receives this
 * call's device status (MLA_OK, MLA_ERR_BAD_TABLE, MLA_ERR_BAD_SEQLEN or
 * MLA_ERR_TIMEOUT) when the call's work has run.
 *
 * Limit: the scratch of one call is about (B + clusters - 1) * Lq*H * 2 KiB
 * (clusters = CTA pairs that fit on the GPU, e.g. 76 on a GB300 at Lq*H <=
 * 128); if that exceeds 32 MiB the call returns MLA_ERR_WORKSPACE and does
 * nothing.  The first call on a device looks up the array's device address;
 * make that first call before any stream capture.  All calls on a device
 * share the array (each call clears and rewrites what it uses), so calls that
 * may overlap on the GPU — unordered streams, several host threads — race.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
int mla_decode_attend_noalloc(const mla_dims* dims, const void* q_cat,
                              const void* kv_cache, const int32_t* block_table,
                              const int32_t* seq_lens, void* o_lat, float* lse,
                              int* device_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
