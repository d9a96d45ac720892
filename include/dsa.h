/*
 * dsa.h -- C ABI of libdsa.so: the gated DSA attention step on one GB300 (sm_103a).
 *
 * The step, per query token t of a sequence:
 *   1. lightning indexer: score every causal key s <= t,
 *        I[t,s] = sum_j w[t,j] * max(0, q_I[t,j,:] . k_I[s,:])
 *      (BF16 inputs, FP32 accumulation) and keep the top-k keys;
 *   2. sparse MLA in latent space over the kept rows only:
 *        z_s = scale * q_lat[t,h,:] . KV[s,:]   (576 = 512 c_kv + 64 unrotated k_pe)
 *        o_lat[t,h,:] = softmax_s(z) . KV[s, 0:512],  lse[t,h] = log sum_s exp(z_s);
 *   3. output gate: out[t, h*dv+e] = sigmoid(x[t] . W_g[h*dv+e]) * (W_uv[h,e,:] . o_lat[t,h,:]).
 *
 * Sources (page title, section):
 *   "Kimi-K3.1-Pro" (NeMo AutoModel model coverage), Implementation Limits:
 *     bullet 1 (a fused indexer yields top-k coordinates; sparse MLA attends
 *     directly to the selected latent KV), bullet 2 (BF16 indexer projections,
 *     FP32 score accumulation, all causal keys scanned, no per-head K/V
 *     expansion), bullet 4 (<= 2,048 valid tokens keep every causal key),
 *     closing paragraph (the output gate is kept; packed documents must be
 *     contiguous).
 *   "Kimi K3.1 Pro" (archdiff, attn-gate): summary (top-2,048 DSA indexer in
 *     the gated MLA layers, no positional encoding); blueprint entries
 *     "LayerNorm on the indexer key" and the output gate sigma(x W_g) (.) o.
 *   "nemo_automodel.components.models.kimi_k3" (v0.4 API), KimiK3TextConfig:
 *     num_attention_heads 96, kv_lora_rank 512, qk_nope_head_dim 128,
 *     qk_rope_head_dim 64 (softmax scale 1/sqrt(192)), v_head_dim 128,
 *     hidden_size 7168, mla_use_nope, mla_use_output_gate.
 *   The indexer's head count, head dim and head-weighted ReLU form are not on
 *   the pages; this library adopts the form above (64 heads x 128, or 4 x 64).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; BF16 values
 *     are passed as uint16_t bit patterns.  Arrays are dense row-major in the
 *     shapes given.  The library allocates, frees and synchronises nothing
 *     (except dsa_read_device_status, which synchronises `stream`), keeps no
 *     global state and launches only on `stream` (NULL = legacy default stream).
 *   - Causality: query i of sequence b sits at absolute position
 *     q_start[b] + i and sees keys 0 .. q_start[b] + i.  q_start and kv_len are
 *     device int32 arrays of length B with kv_len[b] >= q_start[b] + Tq and
 *     kv_len[b] <= max_kv_len.  Single prefill: q_start = 0, kv_len = T.
 *     Chunk c of a chunked prefill: q_start = c*C, kv_len = (c+1)*C.
 *     Decode: Tq = 1, q_start = L-1, kv_len = L (the new token's rows are
 *     already in the cache).  One contiguous document per sequence.
 *   - Workspace: caller-owned device memory of at least dsa_workspace_bytes()
 *     bytes, 256-byte aligned, prepared once by dsa_workspace_init().  Its
 *     first 256 bytes hold a sticky device status word.  One workspace must
 *     not be used by two calls that may run concurrently.
 *   - Errors: arguments are checked on the host before any launch and a
 *     failing check returns DSA_ERR_INVALID_ARGUMENT / DSA_ERR_UNSUPPORTED /
 *     DSA_ERR_WORKSPACE_TOO_SMALL with nothing launched.  A failed launch
 *     returns DSA_ERR_CUDA.  Conditions only the device can see (an index out
 *     of range or not causal, a page id outside the pool, inconsistent
 *     q_start/kv_len, a wait that ran out of time) are recorded in the status
 *     word and read back with dsa_read_device_status(); the affected rows are
 *     skipped, never dereferenced.  Kernels never trap.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* dsa_stream_t;

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARGUMENT = 1,  /* null pointer, bad size, misaligned buffer */
  DSA_ERR_UNSUPPORTED = 2,       /* dims or page size this build does not compile */
  DSA_ERR_CUDA = 3,              /* a CUDA runtime call or launch failed */
  DSA_ERR_DEVICE_TIMEOUT = 4,    /* device: a bounded wait ran out */
  DSA_ERR_BAD_INDEX = 5,         /* device: index / page id / length out of range */
  DSA_ERR_WORKSPACE_TOO_SMALL = 6
} dsa_status_t;

/*
 * A store of per-token rows (indexer keys: width D_I; latent KV: width 576),
 * BF16, either contiguous or paged.
 *   contiguous (block_table == NULL): base = [B, seq_stride, width]; row s of
 *     sequence b is base + (b*seq_stride + s)*width.  seq_stride >= max_kv_len.
 *   paged: base = pool [num_pages, page_size, width]; row s of sequence b is
 *     pool[block_table[b*max_pages + s/page_size]][s % page_size].
 *     block_table is a device int32 array [B, max_pages]; page_size must be 64;
 *     entries used by a call must lie in [0, num_pages) (checked on device).
 * base must be 16-byte aligned.
 */
typedef struct {
  const void* base;
  int64_t seq_stride;
  const int32_t* block_table;
  int32_t max_pages;
  int32_t page_size;
  int32_t num_pages;
} dsa_rows_t;

typedef enum {
  DSA_OP_INDEXER_TOPK = 0,
  DSA_OP_SPARSE_MLA = 1,
  DSA_OP_GATE = 2,
  DSA_OP_CACHE_APPEND = 3,
  DSA_OP_SPARSE_MLA_BWD = 4
} dsa_op_t;

/* Bytes of workspace an op needs for the given sizes (heads = H_I for the
 * indexer, H for sparse MLA, ignored for the gate).  Always >= 256. */
size_t dsa_workspace_bytes(dsa_op_t op, int B, int Tq, int max_kv_len, int heads, int topk);

/* Zero the status header of a workspace (asynchronous on `stream`). */
dsa_status_t dsa_workspace_init(void* workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * Lightning indexer + top-k ("Kimi-K3.1-Pro", Implementation Limits, bullets
 * 1, 2 and 4; "Kimi K3.1 Pro" archdiff summary: top-2,048).
 *   q_idx  [B, Tq, H_I, D_I] BF16   indexer queries
 *   w      [B, Tq, H_I]      BF16   per-head weights (any sign)
 *   k_idx  rows of width D_I BF16   LayerNorm'd indexer keys
 *   out_idx[B, Tq, topk]     int32  written: for a query at position t, exactly
 *          min(t+1, topk) distinct key positions in [0, t], in unspecified
 *          order, followed by -1 padding.  Among keys with equal scores at the
 *          cut, which ones are kept is unspecified.
 * Supported: (H_I, D_I) in {(64,128), (4,64)}; 1 <= topk <= 2048, topk a
 * multiple of 4; Tq >= 1.  Tq == 1 selects the decode kernels (key ranges
 * split across the GPU, a linear score vector per request in the workspace,
 * then a radix select); Tq > 1 the fused prefill kernel, which keeps every
 * score on chip and only the candidates above each query's running threshold
 * in per-CTA buffers of the workspace (at 64 heads: min(SMs, B * ceil(Tq/4))
 * CTAs x 4 queries x 8,192 candidates x 8 bytes, about 38 MiB on 152 SMs;
 * dsa_workspace_bytes gives the exact figure).
 */
dsa_status_t dsa_indexer_topk(const uint16_t* q_idx, const uint16_t* w, const dsa_rows_t* k_idx,
                              const int32_t* q_start, const int32_t* kv_len, int B, int Tq,
                              int H_I, int D_I, int max_kv_len, int topk, int32_t* out_idx,
                              void* workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * Sparse MLA forward in latent space ("Kimi-K3.1-Pro", Implementation Limits,
 * bullets 1-2; KimiK3TextConfig dims; no rotation of the 64 k_pe dims).
 *   q_lat [B, Tq, H, 576] BF16   absorbed queries ([W_UK^T q_nope | q_pe])
 *   kv    rows of width 576 BF16 latent cache ([c_kv(512) | k_pe(64)])
 *   idx   [B, Tq, topk] int32    key positions; -1 entries are skipped; any
 *         other entry must satisfy 0 <= s <= t (else BAD_INDEX, entry skipped)
 *   scale                        softmax scale (1/sqrt(192) for this model)
 *   o_lat [B, Tq, H, 512] BF16   softmax-weighted sum of KV[s, 0:512]
 *   lse   [B, Tq, H] float or NULL   natural-log log-sum-exp of the logits
 * A query with no valid index gets o_lat = 0 and lse = -inf.
 * Supported: H in {8, 96}; 1 <= topk <= 2048.
 */
dsa_status_t sparse_mla_fwd(const uint16_t* q_lat, const dsa_rows_t* kv, const int32_t* idx,
                            const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int H,
                            int topk, int max_kv_len, float scale, uint16_t* o_lat, float* lse,
                            void* workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * sparse_mla_fwd with a learnable attention sink ("Kimi K3.1 Pro" archdiff
 * blueprint, "Output gate + sink"; whether K3.1 uses it is not settled by the
 * pages, so it is a separate entry point).  Same arguments as sparse_mla_fwd
 * plus
 *   sink [H] FP32 (device)   per-head sink logit in natural-log units
 * which joins each head's softmax denominator with no value row:
 *   o = sum_s e^{z_s} v_s / (e^{sink} + sum_s e^{z_s}),
 *   lse = log(e^{sink} + sum_s e^{z_s})
 * A query with no valid entry gets o = 0 and lse = sink.  sink = -inf for a head
 * gives sparse_mla_fwd's result for it.  sink must not be NULL.
 */
dsa_status_t sparse_mla_fwd_sink(const uint16_t* q_lat, const dsa_rows_t* kv, const int32_t* idx,
                                 const int32_t* q_start, const int32_t* kv_len, int B, int Tq,
                                 int H, int topk, int max_kv_len, float scale, const float* sink,
                                 uint16_t* o_lat, float* lse, void* workspace, size_t ws_bytes,
                                 dsa_stream_t stream);

/*
 * Sparse MLA backward ("Kimi-K3.1-Pro", Implementation Limits: attention over
 * the selected rows only, bullets 1-2; a native 96-head backward, the paragraph
 * after bullet 4; hard top-k passes no gradient to the indexer, bullet 3, so
 * idx is a constant).  The gradient of sum(d_o * o_lat) given the forward's
 * outputs:
 *   p_j  = exp(scale * q . kv[s_j] - lse),  dp_j = d_o . kv[s_j, 0:512]
 *   dz_j = p_j (dp_j - D),  D = d_o . o_lat
 *   dq   = scale * sum_j dz_j kv[s_j, 0:576]                       (written)
 *   dkv[s_j, 0:576] += scale * dz_j q,  dkv[s_j, 0:512] += p_j d_o  (added)
 * Arguments as for sparse_mla_fwd, plus
 *   o_lat, lse          the forward's outputs for the same inputs (those of
 *                       sparse_mla_fwd_sink serve too: the sink carries no value
 *                       and depends on neither q nor kv, so only lse sees it)
 *   d_o   [B,Tq,H,512]  BF16   upstream gradient of o_lat
 *   dq    [B,Tq,H,576]  FP32   written; a query with no valid entry gets 0
 *   dkv                 FP32   rows of 576 numbered like kv's rows
 *                              ([B, seq_stride, 576] or [num_pages, 64, 576]),
 *                              16-byte aligned, ADDED to (zero it first).
 *                              Additions come from many queries in no fixed
 *                              order, so the FP32 rounding varies run to run.
 * -1 entries are skipped; other invalid entries raise DSA_ERR_BAD_INDEX and are
 * skipped.  Supported: H <= 128, topk <= 2048.  All products take BF16
 * operands with FP32 accumulation; p and scale * dz are rounded to BF16 for them.
 * Workspace: the 256-byte status header is required.
 *   - With H = 96 and a workspace of dsa_workspace_bytes(DSA_OP_SPARSE_MLA_BWD,
 *     B, Tq, max_kv_len, 96, topk) bytes (the header plus P and dz of up to 512
 *     queries: min(B*Tq, 512) * 96 * ceil(topk/128)*128 * 4 bytes), and d_o,
 *     o_lat, dq 16-byte aligned, the tcgen05 kernels run (queries in chunks of
 *     as many as the workspace holds, at least one).
 *   - Otherwise the warp-level tensor-core MMA kernels run.
 */
dsa_status_t sparse_mla_bwd(const uint16_t* q_lat, const dsa_rows_t* kv, const int32_t* idx,
                            const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int H,
                            int topk, int max_kv_len, float scale, const uint16_t* o_lat,
                            const float* lse, const uint16_t* d_o, float* dq, float* dkv,
                            void* workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * Output gate ("Kimi K3.1 Pro" archdiff blueprint: sigma(x W_g) (.) o;
 * "Kimi-K3.1-Pro", Implementation Limits, closing paragraph: the gate is kept;
 * KimiK3TextConfig mla_use_output_gate, v_head_dim 128).
 *   x     [N, hid] BF16          layer input
 *   W_g   [H*dv, hid] BF16       gate weight, one row per output feature
 *   o_lat [N, H, 512] BF16       sparse MLA output
 *   W_uv  [H, dv, 512] BF16      per-head value up-projection
 *   out   [N, H*dv] BF16         sigmoid(x . W_g[c]) * (W_uv[h,e] . o_lat[n,h]), c = h*dv+e
 * Supported: dv == 128, hid % 64 == 0, H >= 1; N >= 1.
 */
dsa_status_t mla_gate_apply(const uint16_t* x, const uint16_t* W_g, const uint16_t* o_lat,
                            const uint16_t* W_uv, int N, int hid, int H, int dv, uint16_t* out,
                            void* workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * The step just before the indexer: LayerNorm of the new tokens' indexer keys
 * and their append, with the new latent rows, to the two caches ("Kimi K3.1
 * Pro" archdiff blueprint: LayerNorm on the indexer key; eps is
 * KimiK3TextConfig rms_norm_eps, 1e-5).  One call covers a decode step (Tq = 1)
 * or a prefill chunk.
 *   k_pre    [B, Tq, D_I] FP32   the new tokens' raw indexer keys
 *   kv_new   [B, Tq, 576] BF16   their latent rows (c_kv then k_pe), copied as is
 *   k_cache  rows of width D_I   row q_start[b]+i of sequence b is written with
 *            BF16 (round to nearest even) of (x - mean(x)) / sqrt(var(x) + eps),
 *            x = k_pre[b,i,:], var the population variance (unit gain, zero
 *            bias), computed in FP32
 *   kv_cache rows of width 576   row q_start[b]+i of sequence b := kv_new[b,i,:]
 *   q_start  [B] int32 (device)  position of sequence b's first new token
 * The caches' base pointers are written through: dsa_rows_t declares them const
 * for the read-side calls that share it.  A row that does not exist -- a
 * negative position, a page beyond max_pages, a block-table entry outside
 * [0, num_pages), or past seq_stride when contiguous -- is not written and is
 * recorded as DSA_ERR_BAD_INDEX in the workspace status word.
 * Supported: D_I in {64, 128}; B, Tq >= 1; eps >= 0 and finite.  Workspace:
 * dsa_workspace_bytes(DSA_OP_CACHE_APPEND, ...) = the 256-byte status header.
 */
dsa_status_t dsa_cache_append(const float* k_pre, const uint16_t* kv_new,
                              const dsa_rows_t* k_cache, const dsa_rows_t* kv_cache,
                              const int32_t* q_start, int B, int Tq, int D_I, float eps,
                              void* workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * FP8 indexer variant.  "Kimi-K3.1-Pro" (NeMo AutoModel), Implementation
 * Limits, bullet 2, contrasts its BF16 indexer with the FP8 indexer that some
 * serving kernels use.  The pages give nothing more, so the format is this
 * library's reading:
 *   - Codes are E4M3: sign, 4 exponent bits with bias 7 and 3 mantissa bits.
 *     The largest finite value is 448 and there is no infinity.
 *   - Each row of D values (one indexer key, or one head of one query) has one
 *     FP32 scale and stands for scale * decode(code).
 *
 * dsa_quant_fp8 quantizes BF16 rows, exactly as follows:
 *   scale[r]  = max(max_d |x[r,d]|, 2^-100) / 448
 *               (FP32 division, rounded to nearest)
 *   code[r,d] = E4M3(x[r,d] * (1 / scale[r]))
 *               (FP32 reciprocal and product, each rounded to nearest;
 *                E4M3 rounding to nearest even, saturating at +-448)
 *   x     [n_rows, D] BF16
 *   codes [n_rows, D] uint8
 *   scale [n_rows]    FP32
 * Supported: D in {64, 128}.
 * Alignment: x 8 bytes, codes and scale 4 bytes.
 * Nothing can fail on the device, so the call takes no workspace.
 */
dsa_status_t dsa_quant_fp8(const uint16_t* x, int64_t n_rows, int D, uint8_t* codes, float* scale,
                           dsa_stream_t stream);

/*
 * dsa_cache_append with the indexer key stored in FP8.  Each key becomes
 * D_I bytes of codes, written to k_codes (a row store of D_I-byte rows), plus
 * one FP32 scale at the same row of k_scale.
 *   k_scale  is laid out like k_codes' rows:
 *              contiguous: [B, seq_stride]
 *              paged:      [num_pages, 64], through the same block table
 *   values   dsa_quant_fp8 applied to the BF16 row that dsa_cache_append
 *            would have written
 * The latent row, the checks and the device-side errors are those of
 * dsa_cache_append.
 */
dsa_status_t dsa_cache_append_fp8(const float* k_pre, const uint16_t* kv_new,
                                  const dsa_rows_t* k_codes, float* k_scale,
                                  const dsa_rows_t* kv_cache, const int32_t* q_start, int B,
                                  int Tq, int D_I, float eps, void* workspace, size_t ws_bytes,
                                  dsa_stream_t stream);

/*
 * dsa_indexer_topk on FP8 operands.
 *   q_codes [B, Tq, H_I, D_I] uint8   E4M3 query codes
 *   q_scale [B, Tq, H_I]      FP32    one scale per query head
 *   w       [B, Tq, H_I]      BF16    per-head weights
 *   k_codes                           rows of D_I bytes of E4M3 key codes
 *   k_scale                           FP32, laid out like k_codes' rows
 *                                     (see dsa_cache_append_fp8); 16-byte
 *                                     aligned
 * The score of the dequantised rows is
 *   I[t,s] = sum_j w[t,j] * max(0, (q_scale[t,j] q[t,j]) . (k_scale[s] k[s]))
 *          = k_scale[s] * sum_j (w[t,j] q_scale[t,j]) * max(0, q[t,j] . k[s])
 * The codes' dot products are FP32 tensor-core accumulations of exact E4M3
 * products.  Output, workspace and errors are as for dsa_indexer_topk.
 * Supported:
 *   - H_I = 64, D_I = 128; Tq == 1 takes the decode kernels, Tq > 1 the fused
 *     prefill kernel, as for dsa_indexer_topk;
 *   - contiguous key stores need seq_stride % 4 == 0.
 */
dsa_status_t dsa_indexer_topk_fp8(const uint8_t* q_codes, const float* q_scale, const uint16_t* w,
                                  const dsa_rows_t* k_codes, const float* k_scale,
                                  const int32_t* q_start, const int32_t* kv_len, int B, int Tq,
                                  int H_I, int D_I, int max_kv_len, int topk, int32_t* out_idx,
                                  void* workspace, size_t ws_bytes, dsa_stream_t stream);

/*
 * sparse_mla_fwd_noalloc -- sparse_mla_fwd for callers that cannot allocate
 * device memory.  The pages have no counterpart to this entry point; it exists
 * for deployment only.
 *
 * Who needs it: code that runs inside a host framework which owns all device
 * memory (an inference server that hands its memory to a fixed pool at
 * start-up, a plugin interface that passes tensors in and out but offers no
 * scratch), where this call may not reach cudaMalloc.  It takes the same
 * arguments and gives the same results as sparse_mla_fwd, with no workspace:
 *   - Scratch (the split-K partial results used when B*Tq is below the SM
 *     count) lives in one fixed 32 MiB array of device memory inside this
 *     library, held by every GPU that loads the library until the process
 *     exits.  A split launch needs B*Tq*splits*H*(512*2 + 4) + 256 bytes, and
 *     the library keeps B*Tq*splits at or below the SM count: with 96 heads
 *     every split fits on parts with up to about 340 SMs.  Larger needs are
 *     rejected with DSA_ERR_WORKSPACE_TOO_SMALL before anything is launched;
 *     that is the only failure this fixed size adds.  The call allocates and
 *     frees nothing.
 *   - Every call looks up that array's device address on the caller's
 *     current device (a lookup, no allocation).  The first call on a device
 *     also loads this library's device code there; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the array and it keeps the last call's
 *     contents: two calls whose kernels may overlap on the GPU (different
 *     streams without ordering) race on it.  Serialise them.
 *   - device_status: NULL, or a caller-owned device array of 3 uint32 that
 *     starts at zero; device-side errors (bad index, bad page id, a wait that
 *     ran out) are recorded there as in the workspace status word.  With NULL
 *     they are recorded in the array's own header, which each call clears, and
 *     cannot be read back.
 */
dsa_status_t sparse_mla_fwd_noalloc(const uint16_t* q_lat, const dsa_rows_t* kv,
                                    const int32_t* idx, const int32_t* q_start,
                                    const int32_t* kv_len, int B, int Tq, int H, int topk,
                                    int max_kv_len, float scale, uint16_t* o_lat, float* lse,
                                    uint32_t* device_status, dsa_stream_t stream);

/* Synchronise `stream`, return the first device-side error recorded in the
 * workspace (DSA_OK if none) and clear it.  `where` / `detail` (nullable)
 * receive the site tag and detail value. */
dsa_status_t dsa_read_device_status(void* workspace, dsa_stream_t stream, uint32_t* where,
                                    uint32_t* detail);

/*
 * Failure-path self-test (no counterpart on the pages): launch one CTA whose
 * bounded mbarrier wait is never satisfied, so it gives up after limit_ns
 * (at most 200 ms), records DSA_ERR_DEVICE_TIMEOUT in the workspace status
 * word and returns.  Read the result with dsa_read_device_status().  This is
 * the same bounded wait every kernel uses; no kernel traps or spins forever.
 */
dsa_status_t dsa_selftest_wait_timeout(void* workspace, size_t ws_bytes, uint64_t limit_ns,
                                       dsa_stream_t stream);

/* Static string for a status code. */
const char* dsa_status_string(dsa_status_t status);

/* Library ABI version (incremented on incompatible changes). */
int dsa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
