/*
 * k8v4.h -- C ABI of the k8v4 quantized paged KV cache and its fused attention
 * for one GB300 GPU (sm_103a).
 *
 * The cache format is the hybrid "k8v4" KV cache of the pull request
 * "--kv k8v4: hybrid KV cache -- INT8 K + Hadamard-rotated Q4_0 V (816 B/cell)"
 * (section "What"): K is stored as symmetric INT8, V is rotated per head by the
 * orthonormal 256-point Walsh-Hadamard transform and stored as Q4_0, 816 bytes
 * per cell at 2 KV heads x head_dim 256.  Attention reads the compressed cache in
 * three modes (section "How": one fused decode/prefill/verify attention over the
 * hybrid layout; q is not rotated, the output is computed in rotated space and
 * rotated back).  The block of a page holds three byte runs -- K codes, K
 * scales, V q4_0 -- as in "kv: --kv k8v4 streams with --kv-resident" (section
 * "How").
 *
 * Conventions for every call:
 *  - All array arguments are DEVICE pointers owned by the caller (the library
 *    never allocates; scratch lives in the caller's workspace), except where
 *    a call allows page-locked host memory.  `stream` is a cudaStream_t
 *    (NULL = legacy default stream).  Calls are asynchronous.
 *  - Arguments are validated on the host before any launch; a call that fails
 *    validation launches nothing and returns a negative k8v4_status.
 *  - Values that live in device memory (positions, lengths, page-table entries)
 *    are checked by the kernels: an out-of-range page id, position or length is
 *    skipped (never dereferenced) and recorded in a device status word that
 *    k8v4_last_device_status() returns.  No kernel traps or spins.
 *  - The library never calls exit() and never throws across the ABI.
 *  - At its first call on a device the library looks up, with that device
 *    current, the device addresses of its own device variables (the status
 *    word below) and keeps them for the life of the process; do not use the
 *    library on a device after cudaDeviceReset() on it.
 *  - Query head h reads KV head h / 8 (GQA group of 8 query heads).
 *
 * Page layout (per page of P cells and H KV heads; r = slot * H + head):
 *   format K8V4 (408 B per cell and head):
 *     K codes   int8 [P][H][256]        at 0
 *     K scales  f32  [P][H][2]          at 256*H*P    (one per 128-lane half)
 *     V nibbles u8   [P][H][8][16]      at 264*H*P    (byte j of a block:
 *                                                      code j | code j+16 << 4)
 *     V scales  f16  [P][H][8]          at 392*H*P
 *   format INT8 (the 1,056 B/cell comparison arm, 528 B per cell and head):
 *     K codes [P][H][256] at 0, K scales [P][H][2] f32 at 256*H*P,
 *     V codes [P][H][256] at 264*H*P, V scales [P][H][2] f32 at 520*H*P.
 *   format Q4 (the 576 B/cell q4_0 arm, 288 B per cell and head; K and V both
 *   rotated Q4_0, nibble bytes as for the V of K8V4):
 *     K nibbles [P][H][8][16] at 0, K scales f16 [P][H][8] at 128*H*P,
 *     V nibbles [P][H][8][16] at 144*H*P, V scales f16 [P][H][8] at 272*H*P.
 *   Cell c of sequence b lives in page page_table[b * max_pages + c / P],
 *   slot c % P.
 *
 * Arithmetic (bit-exact; where the pages leave a step open the plainest
 * reading is taken and stated here):
 *   K half (128 lanes): s = absmax / 127 (fp32 division), code =
 *     clamp(rint_even(x / s), -127, 127); s == 0 -> codes 0.
 *   V: y = RN_fp32((H_256 x) / 16), Sylvester H, the sum exact; per 32-block:
 *     m = element of largest |y| (first index on ties), d = fp16_RN(m / -8),
 *     code = clamp(rint_even(y / d) + 8, 0, 15); d == 0 -> codes 8.
 *   Attention: out = softmax(sm_scale * q . Khat) . Vhat, Khat = code * s,
 *     Vhat = (H/16) * ((code - 8) * d); fp32 result.
 *   Q4 format: K is rotated and quantised exactly as V, Khat = (H/16) *
 *     ((code - 8) * d); the scores are computed as ((H/16) q) . ((code - 8) * d)
 *     (H/16 is symmetric and orthogonal, so the two are equal).
 */
#ifndef K8V4_H
#define K8V4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  Every entry point returns one of these. */
typedef enum {
  K8V4_OK = 0,
  K8V4_EINVAL = -1,  /* a NULL pointer, a bad enum, a size or shape out of range */
  K8V4_ERANGE = -2,  /* (device) a position, length or page id out of range */
  K8V4_EALIGN = -3,  /* a pointer not aligned as documented */
  K8V4_ECUDA = -4,   /* a CUDA runtime call failed (launch, attribute, ...) */
  K8V4_EDEVICE = -5, /* no sm_103 device, or the library was built for another */
  K8V4_ENOSPACE = -6 /* the caller's workspace is smaller than required */
} k8v4_status;

/* Element type of K/V/q inputs. */
typedef enum { K8V4_F32 = 0, K8V4_BF16 = 1 } k8v4_dtype;

/* Cache format.  3 is the number the streaming PR ("How") gives the hybrid
 * format's enumerator kKvHybrid; 1 is the all-INT8 comparison format and 2
 * the all-q4_0 one (the pages give those two no numbers; these are this
 * library's). */
typedef enum { K8V4_FORMAT_INT8 = 1, K8V4_FORMAT_Q4 = 2, K8V4_FORMAT_K8V4 = 3 } k8v4_format;

/* Descriptor of a caller-owned paged cache (plain data, no ownership). */
typedef struct {
  void* pages;        /* device; n_pages * page_size * k8v4_bytes_per_cell() bytes,
                         256-byte aligned */
  int64_t n_pages;    /* number of physical pages, >= 1 */
  int32_t page_size;  /* P, cells per page: a multiple of 16, 16..4096 */
  int32_t n_kv_heads; /* H, 1..8 */
  int32_t head_dim;   /* must be 256 */
  int32_t format;     /* k8v4_format */
} k8v4_cache;

/* Bytes per cell (all H heads) of a format: 816 for K8V4, 1,056 for INT8 and
 * 576 for Q4 at H = 2 (the three sizes the k8v4 PR compares in "What").
 * Returns 0 for an unknown format or H outside 1..8. */
size_t k8v4_bytes_per_cell(int32_t format, int32_t n_kv_heads);

/* Human-readable name of a status code (static string). */
const char* k8v4_status_string(int status);

/* K8V4_OK if the current device is an sm_103 part this library was built for,
 * else K8V4_EDEVICE. */
int k8v4_device_check(void);

/* Quantise n_tok new tokens per sequence and write them through the page table
 * (the append of the k8v4 PR, "How": K to INT8, V rotated then Q4_0 -- in
 * the Q4 format K is rotated and quantised like V; the
 * per-step decode, verify-window and prompt appends of the streaming PR are all
 * this call with different n_tok).
 *   page_table: int32 [n_seqs][max_pages], physical page ids in [0, n_pages).
 *   pos:        int64 [n_seqs], first logical cell written for sequence b;
 *               cells pos[b] .. pos[b] + n_tok - 1 are written.
 *   k, v:       [n_seqs][n_tok][H][256] of `dtype` (K8V4_F32 or K8V4_BF16),
 *               16-byte aligned, finite values with |x| < 2^100.
 * Device-side: a cell whose page index reaches max_pages or whose page id is
 * out of range is skipped and K8V4_ERANGE is recorded.
 * The exact rotation has a rarely-taken slow path for vectors whose values span
 * more than 2^55 in magnitude; the result is the same either way. */
int kv_append_k8v4(const k8v4_cache* cache, const int32_t* page_table, int64_t max_pages, int32_t n_seqs,
                   const int64_t* pos, int32_t n_tok, const void* k, const void* v, int32_t dtype,
                   void* stream);

/* Workspace bytes attn_k8v4_decode / attn_k8v4_verify need for a launch with
 * these host-side bounds (the split-K partial results). */
size_t attn_k8v4_workspace_bytes(const k8v4_cache* cache, int32_t n_seqs, int32_t n_q_per_seq,
                                 int32_t max_seq_len);

/* Decode attention: one query (16 heads at H = 2) per sequence over its
 * seq_lens[b] visible cells (the step form of the PR's mode-3 attention, "Tests").
 *   q:        [n_seqs][8*H][256] of q_dtype (not rotated), 16-byte aligned.
 *   seq_lens: int32 [n_seqs] (device), each in [0, max_seq_len].
 *   max_seq_len: host-side upper bound of seq_lens, <= max_pages * P; sizes the
 *             split-K grid.  A longer device length is clipped and recorded.
 *   out:      float [n_seqs][8*H][256], the un-rotated attention output.
 *   workspace: >= attn_k8v4_workspace_bytes(cache, n_seqs, 1, max_seq_len)
 *             bytes of device memory, 256-byte aligned.
 * q and out may instead be page-locked host memory that the device addresses
 * directly (cudaHostAlloc, or cudaHostRegister with mapping, under unified
 * addressing): the kernels read q and write out with plain loads and stores
 * across the host link, so a serving loop needs no copy launches of its own;
 * out is complete when the stream reaches the end of the call.
 * A row with zero visible cells outputs zeros.  Works on every format. */
int attn_k8v4_decode(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                     int64_t max_pages, const int32_t* seq_lens, int32_t n_seqs, int32_t max_seq_len,
                     float sm_scale, float* out, void* workspace, size_t workspace_bytes, void* stream);

/* Fused decode step: append each sequence's newest token, then decode.
 * Equivalent to kv_append_k8v4 of one token at position seq_lens[b] - 1 for
 * every sequence followed by attn_k8v4_decode over seq_lens[b] cells (the
 * engine's decode step: the PR's append of the token's K (int8) and rotated V
 * (q4_0), "What"/"How", then its mode-3 attention, "Tests"); the cache bytes
 * written and the output are the same as those two calls'.  The CTA of the
 * split-K grid whose cell range holds the newest cell writes it before any of
 * its warps reads that cell, so the append costs no separate launch.
 *   k_new, v_new: [n_seqs][H][256] of kv_dtype (K8V4_F32 or K8V4_BF16),
 *             16-byte aligned; device memory, or page-locked host memory as
 *             q and out (read with plain loads by the CTA that appends).
 *   seq_lens: int32 [n_seqs] (device), each in [1, max_seq_len] for a sequence
 *             that gets a token (0: no token, zero output); a length past
 *             max_seq_len is clipped, recorded, and its token not written.
 *   Every other argument as attn_k8v4_decode.  A page id of the newest cell
 *   that is out of range is recorded (K8V4_ERANGE) and the token skipped. */
int attn_k8v4_decode_step(const k8v4_cache* cache, const void* q, int32_t q_dtype, const void* k_new,
                          const void* v_new, int32_t kv_dtype, const int32_t* page_table, int64_t max_pages,
                          const int32_t* seq_lens, int32_t n_seqs, int32_t max_seq_len, float sm_scale,
                          float* out, void* workspace, size_t workspace_bytes, void* stream);

/* Decode attention that allocates nothing and takes no workspace.  The pages
 * have no counterpart to this call; it exists for callers that cannot allocate
 * device memory: a host with no device allocator of its own (a plain C program
 * embedding the library on a fixed device budget handed out up front, or a
 * framework whose memory pool already owns all device memory), or a loop that
 * must not call cudaMalloc/cudaFree because cudaFree synchronises the device.
 * Arguments and results are those of attn_k8v4_decode without the workspace.
 * The split-K partials go to a 4 MiB array in the library's own device memory
 * (every GPU that loads the library holds it until the process exits); calls
 * whose attn_k8v4_workspace_bytes(cache, n_seqs, 1, max_seq_len) exceeds 4 MiB
 * are rejected with K8V4_ENOSPACE before any launch.  The first call on a device
 * looks up the array's device address with that device current; make that
 * first call before any stream capture.  All calls share the one array: calls
 * that overlap on the GPU (other streams, other host threads) race and corrupt
 * each other's results, so serialise them.  Nothing in the array has to start
 * at zero: each call writes every partial it reads.  The looked-up address is
 * kept for the life of the process: after cudaDeviceReset() on a device the
 * cached address is stale, so do not call this entry point on that device
 * again in the same process. */
int attn_k8v4_decode_noalloc(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                             int64_t max_pages, const int32_t* seq_lens, int32_t n_seqs, int32_t max_seq_len,
                             float sm_scale, float* out, void* stream);

/* ---------------------------------------------------------------- split across GPUs
 * One long sequence's decode split by cell range over several GPUs (the path
 * the k8v4 PR's engine runs with its multi-GPU split: the PR's header says it
 * sits on the engine release that splits layers across GPUs): GPU r attends over its cells
 * [cell_begin_r, cell_end_r) with attn_k8v4_decode_partial, the partial rows of
 * all GPUs are exchanged (an all-gather of n_seqs * 8H * 260 floats per GPU),
 * and every GPU merges them with attn_k8v4_combine_partials.  The merged result
 * is the decode output over the union of the ranges.
 *
 * Partial row layout (260 floats per (sequence, query head)): o[256], the
 * un-rotated softmax-weighted sum of V relative to 2^m; m, a base-2 exponent at
 * least the row's largest sm_scale * log2(e) * q . Khat over the range (-inf
 * when the range holds no visible cell); l, the sum of 2^(score - m); two
 * unused floats.  For ranges r the output is
 *   sum_r 2^(m_r - M) o_r / sum_r 2^(m_r - M) l_r,  M = max_r m_r. */

/* Workspace bytes attn_k8v4_decode_partial needs for a range of cell_end -
 * cell_begin cells; 0 for a format other than K8V4 or INT8 or a bad range. */
size_t attn_k8v4_partial_workspace_bytes(const k8v4_cache* cache, int32_t n_seqs, int32_t cell_begin,
                                         int32_t cell_end);

/* Decode attention of each sequence's query over its cells [cell_begin,
 * min(cell_end, seq_lens[b])), written as partial rows.
 *   partial:    float [n_seqs][8*H][260], 16-byte aligned (layout above).
 *   cell_begin: a multiple of 16; cell_end >= cell_begin, a multiple of 16 or
 *               >= max_seq_len.
 *   workspace:  >= attn_k8v4_partial_workspace_bytes(cache, n_seqs, cell_begin,
 *               cell_end) bytes, 256-byte aligned.
 * Other arguments as attn_k8v4_decode.  K8V4 and INT8 formats. */
int attn_k8v4_decode_partial(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                             int64_t max_pages, const int32_t* seq_lens, int32_t n_seqs, int32_t max_seq_len,
                             int32_t cell_begin, int32_t cell_end, float sm_scale, float* partial, void* workspace,
                             size_t workspace_bytes, void* stream);

/* Merge gathered partial rows parts[n_parts][n_seqs][n_rows][260] (device)
 * into out[n_seqs][n_rows][256] (device, float): for each row the weighted sum
 * above; a row whose parts all have m = -inf outputs zeros. */
int attn_k8v4_combine_partials(const float* parts, int32_t n_parts, int32_t n_seqs, int32_t n_rows, float* out,
                               void* stream);

/* Verify attention: n_q queries per sequence, query i of sequence b seeing
 * step_arrays[b][i] cells (the batched form with per-query step arrays, as
 * verify uses it, the k8v4 PR "Tests"; for a speculative window of 4 drafts + 1
 * the steps are len-4 .. len).
 *   q: [n_seqs][n_q][8*H][256]; out: float [n_seqs][n_q][8*H][256];
 *   step_arrays: int32 [n_seqs][n_q] (device), each in [0, max_seq_len];
 *   1 <= n_q <= 8.  Works on every format. */
int attn_k8v4_verify(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                     int64_t max_pages, const int32_t* step_arrays, int32_t n_seqs, int32_t n_q,
                     int32_t max_seq_len, float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                     void* stream);

/* Chunked-prefill attention for one sequence on the tensor cores (tcgen05):
 * n_q_tok query tokens, token t seeing step_arrays[t] cells, or, when
 * step_arrays is NULL, the causal count seq_len - n_q_tok + t + 1 (the chunk
 * occupies the last n_q_tok cells of seq_len).
 *   q: bf16 [n_q_tok][8*H][256]; out: float [n_q_tok][8*H][256];
 *   page_table: int32 [max_pages] for the one sequence; seq_len <= max_pages * P.
 * K8V4 format only. */
int attn_k8v4_prefill(const k8v4_cache* cache, const void* q, int32_t q_dtype, const int32_t* page_table,
                      int64_t max_pages, int32_t seq_len, int32_t n_q_tok, const int32_t* step_arrays,
                      float sm_scale, float* out, void* stream);

/* Dequantise cells [start, start + n_cells) of one sequence, for checking (the
 * PR's gather entry points, "Tests": appends and gathers checked bitwise).
 *   k_out:     float [n_cells][H][256] = code * s (Q4 format: RN_fp32((H/16)
 *              ((code - 8) * d)), the exact inverse rotation of the stored K)
 *   v_rot_out: float [n_cells][H][256] = (code - 8) * d (rotated space; for the
 *              INT8 format: code * s, unrotated)
 *   v_out:     NULL or float [n_cells][H][256] = RN_fp32((H/16) v_rot), the
 *              exact inverse rotation (INT8 format: a copy of v_rot_out). */
int kv_dequant_k8v4(const k8v4_cache* cache, const int32_t* page_table, int64_t max_pages, int64_t start,
                    int64_t n_cells, float* k_out, float* v_rot_out, float* v_out, void* stream);

/* ---------------------------------------------------------------- streaming
 * A streamed cache (the streaming PR, "How"): the authoritative copy of every
 * page lives in a host mirror -- a k8v4_cache whose `pages` is page-locked host
 * memory the device can address (cudaHostAlloc, or cudaHostRegister'ed), with
 * the format, P and H of the device cache.  The device cache holds n_resident
 * resident slots (slots 0 .. n_resident - 1) followed by staging slots that a
 * streamed call fills with the pages it misses.  Every writer writes both
 * copies (kv_append_k8v4_mirrored), so a page read from its resident slot and
 * the same page copied from the mirror hold the same bytes, and attention over
 * either is bitwise the same (the PR's "Tests").
 *   slot_of_page: int32 [host n_pages] (device): the resident slot holding host
 *                 page p (0 .. n_resident - 1), or -1 when p is not resident.
 * A host pointer that is not page-locked memory mapped for the current device
 * is rejected with K8V4_EINVAL before any launch. */

/* Append to a streamed cache: page_table holds HOST page ids; every cell is
 * written to its mirror page and, when slot_of_page[page] >= 0, to that device
 * slot as well, from one quantisation (the PR's writers write both halves'
 * host copies, "How").  Other arguments as kv_append_k8v4.  A slot value other
 * than -1 outside [0, dev n_pages) is recorded (K8V4_ERANGE); the mirror is
 * still written. */
int kv_append_k8v4_mirrored(const k8v4_cache* host, const k8v4_cache* dev, const int32_t* slot_of_page,
                            const int32_t* page_table, int64_t max_pages, int32_t n_seqs, const int64_t* pos,
                            int32_t n_tok, const void* k, const void* v, int32_t dtype, void* stream);

/* Workspace bytes of kv_stream_resolve: 16 + 8 * n_seqs * max_pages (the copy
 * list); 0 if n_seqs * max_pages exceeds 2^28. */
size_t kv_stream_workspace_bytes(int32_t n_seqs, int64_t max_pages);

/* The page lookups of one streamed attention call, and the copies of its misses
 * (the PR's block resolve and copy, "How").  Every page that sequence b reads
 * -- page indices below ceil(min(seq_lens[b], max_seq_len) / P) -- is looked
 * up in (sequence, page index) order: a resident page maps to its slot; the
 * r-th miss is copied from the mirror into staging slot n_resident + r.
 *   page_table:     int32 [n_seqs][max_pages], host page ids (device memory).
 *   seq_lens:       int32 [n_seqs] (device), the cells each sequence reads
 *                   (decode: its length; verify: its largest step).
 *   dev_page_table: int32 [n_seqs][max_pages] (device, written): the slot of
 *                   every page read, -1 for entries no cell reaches.
 *   workspace:      >= kv_stream_workspace_bytes(n_seqs, max_pages) bytes,
 *                   16-byte aligned.
 * Then attn_k8v4_decode / attn_k8v4_verify on the device cache with
 * dev_page_table read exactly the bytes of the host pages.  Device-side: a miss
 * with no staging slot left is not copied, its entry is -1 and K8V4_ENOSPACE is
 * recorded; a host page id or slot value out of range gives -1 and
 * K8V4_ERANGE.  A page two sequences share is copied once per miss. */
int kv_stream_resolve(const k8v4_cache* host, const k8v4_cache* dev, const int32_t* slot_of_page,
                      int32_t n_resident, const int32_t* page_table, int64_t max_pages, const int32_t* seq_lens,
                      int32_t n_seqs, int32_t max_seq_len, int32_t* dev_page_table, void* workspace,
                      size_t workspace_bytes, void* stream);

/* Copy whole pages from the host mirror into device slots (all runs of a page):
 * host page pages[i][0] -> slot pages[i][1] for i < n (e.g. to fill the
 * resident window).  pages: int32 [n][2] (device), 8-byte aligned.  An id out of
 * range is recorded (K8V4_ERANGE) and its copy skipped. */
int kv_stream_copy(const k8v4_cache* host, const k8v4_cache* dev, const int32_t* pages, int32_t n, void* stream);

/* Failure-handling diagnostics: the bound, in nanoseconds, of every mbarrier
 * wait in the kernels that use them (TMA-fed decode, tensor-memory prefill and
 * verify); 0 restores each kernel's default (about one second), and a bound
 * under 1000 ns means a single poll with no waiting.  A wait that runs out
 * records K8V4_ECUDA, the kernel releases what it holds and returns; a tiny
 * bound therefore makes such a call fail without harm (the copies and MMAs it
 * already issued are still waited for, with the default bound), which is how
 * the recovery path is tested.  Process-wide; not for production use. */
void k8v4_set_wait_limit_ns(uint32_t ns);

/* Failure-handling diagnostics: nonzero makes every later launch of the
 * TMA-fed decode kernel (attn_k8v4_decode, _decode_step, _decode_noalloc and
 * _decode_partial on the K8V4 and INT8 formats) withhold the copies of one
 * tile: worker 0 of the CTA for split 0, KV head 0, sequence 0 never issues
 * its first tile, so its wait on that stage runs out after the wait bound
 * (k8v4_set_wait_limit_ns) -- a phase that nothing completes -- and the kernel
 * records K8V4_ECUDA, closes that stage itself, waits for its copies in flight
 * and returns.  Zero restores normal operation.  Process-wide; not for
 * production use. */
void k8v4_set_withheld_copy(int32_t on);

/* Synchronise `stream`, return the first device-side error recorded since the
 * last call (K8V4_OK if none) and clear it.  The word is per device and shared
 * by all streams. */
int k8v4_last_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* K8V4_H */
