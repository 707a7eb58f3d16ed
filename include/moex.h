/*
 * moex -- block-quantized GEMV and grouped-MoE expert kernels for one GB300
 * (sm_103a).  C ABI.
 *
 * Sources of the operations (the Strata pull-request pages):
 *   #242  "IQ kernels: decode each weight part once for every column and
 *          entry, bitwise identical" -- What it does: multi-column GEMV,
 *          grouped gate/up and down expert GEMVs.
 *   #1424 "Pascal GP100: a Q8_0 decode GEMV ... and IQ3_XXS / IQ3_S tables
 *          in shared memory" -- What changed: Q8_0 GEMV on q8_1 activations
 *          for 1-8 columns; GGUF blocks repacked into planes with pack /
 *          release ownership.
 *   #1525 "prefill: dense IQ4_XS / Q8_0 to FP16 with 16-byte stores, swiglu
 *          + q8_1 and the MoE combine ... fused" -- Change: SwiGLU fused
 *          with q8_1 of H, the top-k combine, FP16 dequantisation.
 *   #2356 "pf_wmma: a second Volta prompt-expert kernel for IQ2_S gate/up
 *          and IQ4_NL down" -- Summary: FP16 tensor-core prompt experts on
 *          rows sorted by expert, IQ4_NL weights dequantised per tile.
 *
 * Conventions for every call:
 *   - Pointers named *_dev / device planes are device memory owned by the
 *     caller; the library allocates nothing and keeps no per-call state.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously; no call synchronises except
 *     moex_device_status().
 *   - Return value: MOEX_OK, or an error found on the host before anything
 *     is enqueued (MOEX_EINVAL / MOEX_EALIGN / MOEX_EUNSUPPORTED /
 *     MOEX_ENOSPACE), or MOEX_ECUDA if a launch failed.  No call aborts or
 *     throws.  Problems found on the device (a routing id out of range, a
 *     bounded wait that ran out) set bits of a device status word read by
 *     moex_device_status(); the outputs of that call are then undefined.
 *   - K (inputs per row) is a multiple of 32.  Device pointers are 16-byte
 *     aligned unless stated otherwise.
 */
#ifndef MOEX_H
#define MOEX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moex_stream; /* same type as cudaStream_t */

typedef enum moex_status {
  MOEX_OK = 0,
  MOEX_EINVAL = 1,       /* bad argument: null pointer, size out of range */
  MOEX_EALIGN = 2,       /* a pointer or stride breaks the alignment rule */
  MOEX_EUNSUPPORTED = 3, /* format or shape this call does not take */
  MOEX_ECUDA = 4,        /* a CUDA runtime call or launch failed */
  MOEX_ETIMEOUT = 5,     /* device: a bounded wait ran out */
  MOEX_EDEVICE = 6,      /* device: bad input seen by a kernel (routing id) */
  MOEX_ENOSPACE = 7      /* workspace smaller than the *_workspace_bytes query */
} moex_status;

typedef enum moex_fmt {
  MOEX_Q8_0 = 1,   /* 32 int8 + FP16 scale per block; value = d * q        */
  MOEX_IQ4_NL = 2  /* 32 4-bit indices into kvalues_iq4nl + FP16 scale     */
} moex_fmt;

/*
 * A stack of n_mats weight matrices (experts) of rows x K in packed planes
 * (#1424 What changed: GGUF blocks repacked so every load is 16 bytes):
 *   qs     : quant plane, matrix m row r at  qs + (m*rows + r) * qs_row_bytes
 *            Q8_0: K int8 in natural order (qs_row_bytes = K);
 *            IQ4_NL: K/2 bytes, the GGUF 16 index bytes of each block kept
 *            as they are (qs_row_bytes = K/2).
 *   scales : FP16 plane, matrix m row r at scales + (m*rows + r) * sc_row_bytes
 *            with sc_row_bytes = K/32*2 rounded up to a multiple of 16.
 * Both planes are device memory owned by the caller, 16-byte aligned.
 */
typedef struct moex_qweight {
  int32_t fmt;    /* moex_fmt */
  int32_t n_mats; /* >= 1 */
  int64_t rows;   /* rows per matrix, >= 1 */
  int64_t K;      /* inputs per row, multiple of 32 */
  void* qs;
  void* scales;
} moex_qweight;

/* Text of a status code (static storage). */
const char* moex_status_string(int status);

/* ABI version, currently 1. */
int moex_version(void);

/* Byte sizes of the two planes of a (fmt, n_mats, rows, K) weight stack. */
moex_status moex_weight_plane_bytes(int fmt, int64_t n_mats, int64_t rows, int64_t K, size_t* qs_bytes,
                                    size_t* scale_bytes);

/*
 * Repacks GGUF blocks into planes on the device (#1424 What changed:
 * "a device-side GGUF-block -> planes repack").
 *   w            : destination planes (fmt, n_mats, rows, K, qs, scales set).
 *   gguf_blocks  : device, n_mats*rows*(K/32) blocks of 34 (Q8_0) or 18
 *                  (IQ4_NL) bytes, row-major, no alignment requirement.
 * The planes are written; the source is left unchanged.  One-time, not part
 * of the timed path.
 */
moex_status moex_weight_pack(const moex_qweight* w, const void* gguf_blocks, moex_stream stream);

/*
 * q8_1 of FP32 activations (#1525 Change: quantize_mmq_q8_1; #1424: "int8
 * plane plus float scales").  Per 32-value block: d = amax/127 (IEEE FP32
 * division), q = roundf(x/d) (IEEE division, half away from zero),
 * s = d * sum(q); an all-zero block gives d = q = s = 0.
 *   x    : device FP32, column c at x + c*ldx, K values each (ldx >= K, ldx % 4 == 0).
 *   q    : device int8 [ncols][K]     (output)
 *   ds   : device float [ncols][K/32][2] = {d, s} per block (output, 8-byte aligned)
 * 1 <= ncols <= 64.
 */
moex_status moex_quantize_q8_1(const float* x, int64_t K, int ncols, int64_t ldx, int8_t* q, float* ds,
                               moex_stream stream);

/*
 * y[c][r] = sum_b fp32(dw[r,b]) * d_x[c,b] * (sum_i qw[r,32b+i] * qx[c,32b+i])
 * for every row r of the (single) matrix W and every column c of X
 * (#242 What it does; #1424 What changed).  Each weight block is read and
 * decoded once and applied to all columns of a pass; passes take up to 8
 * columns.  Column c of a multi-column call is bitwise equal to a one-column
 * call on column c.
 *   W    : n_mats == 1.
 *   xq   : device int8 [ncols][K] (16-byte aligned) and xds device float
 *          [ncols][K/32][2] (8-byte aligned) as written by moex_quantize_q8_1.
 *   y    : device FP32, column c at y + c*ldy (ldy >= rows).
 * 1 <= ncols <= 64.  Float results agree with the exact value within
 * 1e-5 * sum|w*x| + 1e-6 per element.
 */
moex_status moex_qgemv(const moex_qweight* W, const int8_t* xq, const float* xds, int ncols, float* y,
                       int64_t ldy, moex_stream stream);

/*
 * Diagnostic: the per-block integer dots I[c][r][b] = sum_i qw*qx of
 * moex_qgemv (int32, exact), computed by the same device code.
 *   dots : device int32 [ncols][rows][K/32].   1 <= ncols <= 8.
 */
moex_status moex_qgemv_block_dots(const moex_qweight* W, const int8_t* xq, int ncols, int32_t* dots,
                                  moex_stream stream);

/*
 * Test hook for the failure path of the bounded device waits (no counterpart
 * on the pages: they describe no failure detection).  Launches the
 * shared-memory-ring variant of the one-column moex_qgemv kernel with its
 * copy producer switched off: it issues no copy at all, so every consumer
 * warp's wait for its first weight stage runs out after wait_limit_ns
 * nanoseconds of %globaltimer, sets the "copy-pipeline wait ran out" bit of
 * the device status word and returns.  No copy is in flight when the kernel
 * exits, the context stays usable, and y is left undefined.
 *   Arguments as moex_qgemv with ncols == 1 and K <= 2560;
 *   1e5 <= wait_limit_ns <= 2e9.
 * Afterwards moex_device_status() returns MOEX_ETIMEOUT (and clears the
 * word); the next regular call runs normally.
 */
moex_status moex_debug_qgemv_starved(const moex_qweight* W, const int8_t* xq, const float* xds, int ncols, float* y,
                                     int64_t ldy, uint64_t wait_limit_ns, moex_stream stream);

/*
 * Router: top-k experts of each token's logits (descending logit, ties to the
 * lower expert id) and the softmax over the k selected logits (max
 * subtracted; FP32 expf).
 *   logits : device FP32 [T][E];  ids : device int32 [T][k];  w : device FP32 [T][k].
 * 1 <= k <= 16, k <= E <= 1024.
 */
moex_status moex_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                            moex_stream stream);

/* Workspace bytes of moex_moe_decode for T tokens, top-k, inter size. */
size_t moex_moe_decode_workspace_bytes(int T, int k, int64_t hidden, int64_t inter);

/*
 * The grouped MoE decode layer (#242 What it does: grouped gate/up and down
 * GEMVs over every entry of an expert; #1525 Change: swiglu + q8_1 of H
 * fused, the top-k combine):
 *   xq[t]  = q8_1(x[t]);  gu[j] = W_gu[e_j] . xq[t_j]  (gate rows 0..I-1, up I..2I-1)
 *   H[j]   = silu(g) * u (FP32);  Hq[j] = q8_1(H[j])  (H is never stored)
 *   o[j]   = W_dn[e_j] . Hq[j];   out[t] = sum_{k ascending} w[t,k] * o[(t,k)]
 * Each distinct expert's weights are read once for all of its entries.
 *   gate_up : Q8_0 stack [E][2*inter][hidden];  down : IQ4_NL or Q8_0 stack [E][hidden][inter].
 *   x       : device FP32 [T][hidden];  ids, w : device [T][k] (ids in [0,E)).
 *   out     : device FP32 [T][hidden] (overwritten).
 *   ws      : device workspace of moex_moe_decode_workspace_bytes() bytes.
 * 1 <= T*k <= 64; hidden, inter multiples of 32.  Two kernel launches.
 */
moex_status moex_moe_decode(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                            const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes,
                            moex_stream stream);

/*
 * moex_moe_decode with the residual add fused into the combine (#1525
 * Change: the MoE combine folded into the write of the layer output, no
 * round trip of the combined rows): out[t] = residual[t] + (the combine of
 * moex_moe_decode, summed in slot order first), one FP32 addition.
 *   residual : device FP32 [T][hidden], 16-byte aligned; may be out itself.
 */
moex_status moex_moe_decode_residual(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                                     const int32_t* ids, const float* w, int k, const float* residual, float* out,
                                     void* ws, size_t ws_bytes, moex_stream stream);

/*
 * moex_moe_decode that also writes its intermediates, for staged checking:
 *   gu_dbg : device FP32 [T*k][2*inter] gate/up outputs (may be NULL)
 *   h_dbg  : device FP32 [T*k][inter] H before its q8_1 (may be NULL)
 *   hq_dbg : device int8 [T*k][inter] and hds_dbg FP32 [T*k][inter/32][2]:
 *            copies of Hq (may be NULL)
 */
moex_status moex_moe_decode_debug(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                                  const int32_t* ids, const float* w, int k, float* out, void* ws,
                                  size_t ws_bytes, float* gu_dbg, float* h_dbg, int8_t* hq_dbg, float* hds_dbg,
                                  moex_stream stream);

/* Workspace bytes of moex_moe_prefill for T tokens, top-k, E experts. */
size_t moex_moe_prefill_workspace_bytes(int T, int k, int E, int64_t hidden, int64_t inter);

/*
 * Byte offsets of the prefill workspace's parts, for inspection by tests:
 * offsets[0] counts int32[E] (then the sort's per-segment histograms,
 * per-expert offsets and each entry's sorted row, -1 for an entry left out),
 * [1] order int32[T*k] (entry index of each sorted row),
 * [2] {token, weight bits} int32x2[T*k], [3]/[4] tile lists, [5] totals
 * int32[4] (GEMM 1 tiles, GEMM 2 tiles, placed rows, token tiles), [6] Xs
 * FP16 [T*k][hidden] (gathered rows), [7] Hs FP16
 * [T*k][inter] (SwiGLU output), [8] total.  Xs and Hs store each 32-input
 * block interleaved: position 2j holds input j and 2j+1 input j+16.
 */
moex_status moex_moe_prefill_workspace_layout(int T, int k, int E, int64_t hidden, int64_t inter,
                                              size_t* offsets);

/*
 * The grouped MoE prefill layer on FP16 tensor cores (#2356 Summary: prompt
 * rows sorted by expert, IQ4_NL weights dequantised to FP16 per tile with
 * FP32 sums; #1525 Change: one rounding per dequantised value, SwiGLU
 * between the products, the top-k combine):
 *   rows sorted by expert (stable), Xs = fp16(x), Wh = fp16_rn(d * kvalue)
 *   (IQ4_NL) or fp16_rn(d * q) (Q8_0)
 *   H  = fp16(silu(g) * u),  g, u = Wh_gu[e] . Xs   (FP32 accumulation)
 *   out[t] = sum_k w[t,k] * (Wh_dn[e] . H)          (FP32, summed with
 *            atomic adds: the order of the k terms is not fixed)
 *   gate_up, down : IQ4_NL or Q8_0 stacks (each its own format)
 *            [E][2*inter][hidden], [E][hidden][inter].
 *   x_bf16 : device BF16 [T][hidden];  ids, w : device [T][k] (from
 *            moex_route_topk); out : device FP32 [T][hidden] (overwritten).
 *   ws     : device workspace of moex_moe_prefill_workspace_bytes() bytes.
 * hidden % 128 == 0, inter % 64 == 0, E <= 4096, E * 2 * inter < 2^31.
 * Seven launches (sort: histogram, scan, tiles, scatter; gather; GEMM 1,
 * whose epilogue warps also clear out; GEMM 2); the GEMMs use tcgen05 / TMEM
 * / TMA.  An
 * entry whose id is outside [0, E) is left out of the layer and flagged
 * (MOEX_EDEVICE).
 */
moex_status moex_moe_prefill(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16, int T,
                             const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes,
                             moex_stream stream);

/* Workspace bytes of moex_moe_prefill_q8 for T tokens, top-k, E experts. */
size_t moex_moe_prefill_q8_workspace_bytes(int T, int k, int E, int64_t hidden, int64_t inter);

/*
 * Byte offsets of the integer-route workspace: offsets[0] counts (then the
 * sort's histograms, expert offsets and each entry's sorted row), [1] order
 * int32[T*k], [2] {token,
 * weight bits} int32x2[T*k], [3] first-product tile list, [4] down-product
 * tile list, [5] totals, [6] Xs FP16 [T*k][hidden] (interleaved blocks as in
 * the FP16 route), [7] Hq int8 [T*k][inter] (natural order), [8] {d, s}
 * float32x2 [T*k][inter/32], [9] total.  Rows are in sorted order (order[]).
 */
moex_status moex_moe_prefill_q8_workspace_layout(int T, int k, int E, int64_t hidden, int64_t inter,
                                                 size_t* offsets);

/*
 * The grouped MoE prefill layer on its integer route (#1525 Change: the
 * prompt path's SwiGLU fused with the q8_1 quantisation of H --
 * swiglu_quant writing q8_1 rows -- and the down product as block-integer
 * dots, the "MMQ" route beside the FP16 one):
 *   g, u   = Wh_gu[e] . Xs   on FP16 tensor cores (tcgen05), as moex_moe_prefill
 *   H      = silu(g) * u      (FP32, never rounded to FP16)
 *   Hq, Hd = q8_1(H)          per 32-feature block, in the first product's epilogue
 *   o      = sum_b fp32(dw[r,b]) * Hd[b] * (sum_i qw[r,32b+i] * Hq[32b+i])   (dp4a)
 *   out[t] = sum_k w[t,k] * o[(t,k)]   (FP32 atomic adds: order not fixed)
 * Arguments as moex_moe_prefill (no residual form); ws of
 * moex_moe_prefill_q8_workspace_bytes() bytes.  Eight launches (sort:
 * histogram, scan, two tile lists, scatter; gather, which also clears out;
 * the tcgen05 first product; the dp4a down product).
 */
moex_status moex_moe_prefill_q8(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16, int T,
                                const int32_t* ids, const float* w, int k, float* out, void* ws, size_t ws_bytes,
                                moex_stream stream);

/*
 * moex_moe_prefill_q8 that also writes H, for staged checking:
 *   h_dbg : device FP32 [T*k][inter] in sorted-row order (16-byte aligned),
 *           the values the q8_1 quantiser received.
 */
moex_status moex_moe_prefill_q8_debug(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16,
                                      int T, const int32_t* ids, const float* w, int k, float* out, void* ws,
                                      size_t ws_bytes, float* h_dbg, moex_stream stream);

/* Workspace bytes of moex_dense_prefill for T tokens and a rows x K matrix. */
size_t moex_dense_prefill_workspace_bytes(int T, int64_t rows, int64_t K);

/*
 * Dense prefill product on FP16 tensor cores (#1525 Change: dense weights
 * dequantised to FP16 for the prompt product, one rounding per value; the
 * same tcgen05 kernel as the expert GEMMs, on one matrix and every token):
 *   y[t][r] = sum_i fp16_rn(fp32(d) * kv[r,i]) * fp16_rn(x[t][i])   (FP32 sums)
 *   W   : IQ4_NL or Q8_0, n_mats == 1, rows % 128 == 0, K % 64 == 0.
 *   x   : device BF16 bit patterns [T][K], 16-byte aligned.
 *   y   : device FP32, token t at y + t*ldy (ldy >= rows), fully written.
 *   ws  : device workspace of moex_dense_prefill_workspace_bytes() bytes.
 * Three launches (tile list, BF16 -> FP16 rows, the GEMM).
 */
moex_status moex_dense_prefill(const moex_qweight* W, const uint16_t* x_bf16, int T, float* y, int64_t ldy, void* ws,
                               size_t ws_bytes, moex_stream stream);

/*
 * moex_moe_prefill with the residual add fused (#1525 Change): out starts as
 * residual instead of zero, and the second GEMM adds every weighted expert
 * output to it (the order of those FP32 additions is not fixed).
 *   residual : device FP32 [T][hidden], 16-byte aligned; may be out itself.
 */
moex_status moex_moe_prefill_residual(const moex_qweight* gate_up, const moex_qweight* down, const uint16_t* x_bf16,
                                      int T, const int32_t* ids, const float* w, int k, const float* residual,
                                      float* out, void* ws, size_t ws_bytes, moex_stream stream);

/*
 * moex_moe_decode without a workspace argument, for callers that cannot
 * allocate device memory (code running inside another framework's memory
 * pool with no allocator hook, plug-ins that may not allocate after
 * start-up, decode paths that must never call cudaMalloc).  There is no
 * counterpart on the pages this library follows; it is a convenience of the
 * library.
 *   The workspace is a 512 KiB buffer compiled into the library (a
 *   __device__ array that every GPU loading the library keeps until the
 *   process exits).  Layers whose moex_moe_decode_workspace_bytes() exceeds
 *   512 KiB are rejected with MOEX_ENOSPACE.  Nothing is allocated.
 *   The first call on a device looks up the buffer's device address (with
 *   that device current); make that first call before any stream capture.
 *   Every call on a device uses the same buffer, which keeps the previous
 *   call's contents (nothing in it needs clearing: the layer writes every
 *   byte it reads).  Calls that may overlap on the GPU -- on different
 *   streams, or from several threads -- race on the buffer and must be
 *   serialised by the caller.
 * Arguments and results are those of moex_moe_decode, and so are the
 * argument checks, in the same order: a malformed call returns the status
 * moex_moe_decode would return, and MOEX_ENOSPACE means only that a
 * well-formed layer needs more than the built-in buffer.
 */
moex_status moex_moe_decode_noalloc(const moex_qweight* gate_up, const moex_qweight* down, const float* x, int T,
                                    const int32_t* ids, const float* w, int k, float* out, moex_stream stream);

/*
 * Reads and clears the device status word after synchronising `stream`.
 * *flags receives its bits (1: routing id out of range, 2: copy-pipeline
 * wait ran out, 4: tensor-core wait ran out, 8: bad shape on the device).
 * Returns MOEX_OK when the word was 0, MOEX_EDEVICE / MOEX_ETIMEOUT
 * otherwise, MOEX_ECUDA if the stream reported an error.
 */
moex_status moex_device_status(moex_stream stream, uint32_t* flags);

#ifdef __cplusplus
}
#endif

#endif /* MOEX_H */
