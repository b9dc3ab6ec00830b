/*
 * libengram: the DeepSeek-V4.1 Engram residual-memory hot path on one GB300.
 *
 *   hash -> gather + dequant -> wkv projection -> gate (in place)
 *
 * Sources of the operation (pages, by title and section):
 *   [Atlas] "spark_model::layers::engram_v41" rustdoc: module overview, stages 1-4,
 *           constant ENGRAM_ROW_BYTES.
 *   [NeMo]  "nemo_automodel.components.models.deepseek_v41.engram": DeepseekV41Engram.forward,
 *           DeepseekV41NgramHash.forward, _engram_gate_core.
 *   [vLLM]  "vllm.models.deepseek_v41.common.engram": Engram, EngramLayout, NgramHashState,
 *           ParallelEngramEmbedding.lookup / _engram_lookup_kernel, compute_hash_multipliers,
 *           find_next_prime, _is_prime.
 *
 * Conventions shared by every entry point:
 *   - Pointers named "device" are device memory owned by the caller; the library keeps no
 *     reference after the call returns and (except where stated) allocates nothing.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Work is enqueued on it and
 *     the call returns without synchronising.
 *   - Return value: ENGRAM_OK (0), or a negative code; engram_last_error() then returns a
 *     thread-local message. Arguments are checked on the host before any launch; a failed
 *     check launches nothing.
 *   - Data-dependent faults found on the device (an id outside its range) never trap: the
 *     kernel substitutes the documented value and ORs a bit into the caller's `err_flag`
 *     word (device int32, may be NULL to skip reporting). The caller reads it when it likes.
 *   - T == 0 is a no-op that returns ENGRAM_OK.
 */
#ifndef ENGRAM_H_
#define ENGRAM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ENGRAM_OK 0
#define ENGRAM_EINVAL (-1) /* bad argument (shape, pointer, alignment, format) */
#define ENGRAM_ECUDA (-2)  /* a CUDA call or launch failed */
#define ENGRAM_EDATA (-3)  /* engram_sync_status only: a data-dependent bit is set in err_flag */

/* bits of the device err_flag word */
#define ENGRAM_ERR_RAW_ID 1        /* raw input id outside [0, raw_vocab): used pad_id */
#define ENGRAM_ERR_ROW_ID 2        /* row id outside [0, num_rows): wrote a zero row */
#define ENGRAM_ERR_PIPE_TIMEOUT 4  /* a pipeline wait (GEMM, gate) ran past its time limit */

typedef void* engram_stream_t; /* a cudaStream_t */

/* Table row formats. */
enum EngramTableFmt {
  ENGRAM_TABLE_BF16 = 0,    /* bf16 [rows, head_dim] */
  ENGRAM_TABLE_FP8_E8M0 = 1,/* e4m3 [rows, head_dim] + one E8M0 byte per 32 values [rows, head_dim/32] */
  ENGRAM_TABLE_Q2K = 2      /* one 84-byte Q2_K super-block per 256-wide row [rows, 84] */
};

/* wkv formats (EngramLayerWeights.wkv_format). */
enum EngramWkvFmt {
  ENGRAM_WKV_BF16 = 0,      /* bf16 [N, K] */
  ENGRAM_WKV_MXFP8 = 1      /* e4m3 codes [N, K] + one power-of-two scale byte per 32 along K [N, K/32] */
};

/*
 * Model dimensions ([vLLM] EngramLayout fields; [NeMo] DeepseekV41Engram attributes).
 *   layers           engram layers sharing one hash call (len(engram_layer_ids))
 *   max_ngram        n-gram sizes 2..max_ngram are hashed; lookback depth is max_ngram-1
 *   n_heads          hash heads per n-gram size; C = (max_ngram-1)*n_heads columns
 *   head_dim         D, width of one table row
 *   hidden           H
 *   hc               hc_mult, number of highway streams
 *   raw_vocab        entries of token_map
 *   compressed_vocab V; every compressed id and pad_id lies in [0, V)
 *   pad_id           compressed id that fills unavailable window slots
 *   eps              rms_norm_eps of the two branch norms
 *   clamp            lower clamp of |score| before the signed square root (1e-6)
 */
typedef struct EngramDims {
  int32_t layers, max_ngram, n_heads, head_dim, hidden, hc;
  int32_t raw_vocab, compressed_vocab, pad_id;
  float eps, clamp;
} EngramDims;

const char* engram_last_error(void);
const char* engram_version(void);

/*
 * The synchronous form of the err_flag convention: waits for everything enqueued so far on
 * `stream`, reads the device word err_flag and returns
 *   ENGRAM_OK     the word is 0;
 *   ENGRAM_EDATA  (-3) a data-dependent bit is set: ENGRAM_ERR_RAW_ID (a raw input id outside the
 *                 token map, hashed as pad_id, as [NeMo] DeepseekV41NgramHash.forward pads what it
 *                 cannot look back at) or ENGRAM_ERR_ROW_ID (a row id outside the table, read as a
 *                 zero row, as [vLLM] _engram_lookup_kernel reads the rows a rank does not own).
 *                 The results are defined; the inputs were not what the model expects;
 *   ENGRAM_ECUDA  (-2) ENGRAM_ERR_PIPE_TIMEOUT is set (the results are invalid), or a CUDA call
 *                 failed, including an error left by earlier asynchronous work on the stream.
 * engram_last_error() names the bits. The word is not cleared (the caller owns it).
 *   err_flag  device int32, non-NULL, 4-byte aligned.
 */
int engram_sync_status(const int32_t* err_flag, engram_stream_t stream);

/*
 * Host-side layout ([vLLM] EngramLayout.__init__, find_next_prime, _is_prime).
 * For each layer and each n-gram size the search restarts above vocab_size-1 and takes
 * n_heads successive primes never handed out before in the model. Columns are n-gram size
 * major, head minor. offsets are the exclusive running sum of a layer's primes.
 *   primes_out  host int64 [layers, C]     offsets_out host int64 [layers, C]
 *   rows_out    host int64 [layers]        (table rows a layer needs = sum of its primes)
 * Host memory only, no GPU needed. vocab_size + all primes must stay below 2^32.
 */
int engram_layout(int64_t vocab_size, int32_t layers, int32_t max_ngram, int32_t n_heads,
                  int64_t* primes_out, int64_t* offsets_out, int64_t* rows_out);

/*
 * Stage 1: n-gram hash ids ([NeMo] DeepseekV41NgramHash.forward; [vLLM] NgramHashState.forward;
 * [Atlas] stage 1).
 * For token t, layer l, n-gram size n and head h (column c = (n-2)*n_heads + h):
 *     mix = XOR_{k<n} ( w_k(t) * multipliers[l][k] )        (int64, each product < 2^63)
 *     out = offsets[l][c] + mix mod primes[l][c]
 * where w_k(t) is the compressed id k positions back, or pad_id once the walk back from t
 * meets: a dead position (token_mask 0 or sequence_ids 0; a dead t pads its whole window), a
 * change of sequence_ids between neighbours, the start of t's sequence (cu_seqlens), or, in
 * the lookback row, an entry < 0. lookback_ids[s][i] is the compressed id at position
 * cu_seqlens[s] - (max_ngram-1) + i and belongs to the document of the chunk's first token.
 *   input_ids     device int32 [T] raw tokenizer ids; ids outside [0, raw_vocab) hash as pad_id
 *                 and set ENGRAM_ERR_RAW_ID
 *   cu_seqlens    device int32 [S+1], 0 = cu[0] <= ... <= cu[S] = T; NULL = one sequence [0, T)
 *   sequence_ids  device int32 [T] document ids, 0 = padding; NULL = none
 *   token_mask    device uint8 [T], 0 = image/padding; NULL = all valid
 *   lookback_ids  device int32 [S, max_ngram-1] compressed ids, < 0 = unavailable; NULL = none
 *   token_map     device int32 [raw_vocab] raw -> compressed id
 *   multipliers   device int64 [layers, max_ngram], odd, multiplier * (V-1) < 2^63
 *   primes        device int64 [layers, C]      offsets device int64 [layers, C]
 *   out_ids       device int32 [T, layers, C]   (offsets + primes must fit int32)
 * Requires 2 <= max_ngram <= 8, layers * C <= 256.
 */
int engram_hash(const EngramDims* dims, const int32_t* input_ids, int64_t T,
                const int32_t* cu_seqlens, int32_t S, const int32_t* sequence_ids,
                const uint8_t* token_mask, const int32_t* lookback_ids,
                const int32_t* token_map, const int64_t* multipliers, const int64_t* primes,
                const int64_t* offsets, int32_t* out_ids, int32_t* err_flag,
                engram_stream_t stream);

/*
 * Stage 2: gather rows by id and dequantise to bf16 ([vLLM] _engram_lookup_kernel;
 * [Atlas] stage 2, ENGRAM_ROW_BYTES).
 *   FP8_E8M0: y = bf16_rne( float(e4m3 v) * float(bits = scale_byte << 23) ), one scale per 32.
 *   Q2K:      element e of the 84-byte block (16 B sub-block scale|min<<4, 64 B 2-bit quants,
 *             fp16 d, fp16 dmin): q = (qs[32*(e/128) + e%32] >> 2*((e%128)/32)) & 3,
 *             y = bf16_rne( d*(sc&15)*q - dmin*(sc>>4) ) with sc = scales[e/16].
 *   BF16:     copy.
 * Ids outside [0, num_rows) give a zero row and set ENGRAM_ERR_ROW_ID.
 *   ids          device int32, row t at ids + t*ids_stride_t, C contiguous entries
 *   table        device, format `fmt`, 16-byte aligned (4-byte for Q2K)
 *   scales       device uint8 [num_rows, head_dim/32] for FP8_E8M0, else ignored
 *   out          device bf16 [T, C*head_dim] row-major (row t = C rows of head_dim), 16-byte aligned
 * head_dim: multiple of 32 (FP8), 256 (Q2K), 8 (BF16).
 */
int engram_gather_dequant(int32_t fmt, const int32_t* ids, int64_t ids_stride_t, int64_t T,
                          int32_t C, int32_t head_dim, const void* table, const uint8_t* scales,
                          int64_t num_rows, uint16_t* out, int32_t* err_flag,
                          engram_stream_t stream);

/*
 * Stage 3: wkv projection kv = A * wkv^T ([vLLM] Engram.__init__ (wkv) and Engram.forward;
 * [Atlas] stage 3). bf16 operands, fp32 accumulation on tcgen05 tensor cores, fp32 output
 * (the pages keep kv in the model dtype; fp32 keeps the gate's reductions exact to the
 * accumulator, which matters for the larger Q2_K rows).
 *   A    device bf16 [T, K] row-major       wkv device bf16 [N, K] row-major (nn.Linear layout)
 *   kv   device fp32 [T, N] row-major; columns [j*H, (j+1)*H) are stream j's key, [hc*H, N)
 *        the shared value
 * K % 8 == 0, N % 16 == 0, all three 16-byte aligned.
 *   workspace  device, 256-byte aligned, or NULL. Used only by the stream-K schedule (opt-in,
 *              engram_set_gemm_schedule(2)): with at least engram_project_workspace_bytes(T, K, N)
 *              bytes (one flag per SM), shapes with fewer 256-wide tiles than twice the SM count
 *              split the k-blocks of all tiles evenly over the SMs; a tile cut between CTAs is
 *              summed into kv segment by segment in a fixed order (deterministic results).
 *              Otherwise each CTA runs whole tiles. Nothing in it needs to start at zero.
 * ENGRAM_ERR_PIPE_TIMEOUT in err_flag means the result is invalid; while that bit is set in the
 * word passed, later calls with the same word skip the work.
 */
int engram_project(const uint16_t* A, const uint16_t* wkv, float* kv, int64_t T, int32_t K,
                   int32_t N, void* workspace, size_t ws_bytes, int32_t* err_flag,
                   engram_stream_t stream);

/*
 * The tile plan engram_project (wkv_format ENGRAM_WKV_BF16) or engram_project_mxfp8
 * (ENGRAM_WKV_MXFP8) would launch for a [T, K] x [N, K]^T projection on a GPU with num_sms SMs,
 * under the current tuning knobs. Host only: no GPU is needed or touched. A diagnostic for
 * choosing shapes and knobs. Returns ENGRAM_EINVAL if no plan fits (the launch would refuse too).
 *
 * The tensor cores read a full 128-row token tile from every stage even when fewer rows were
 * loaded (a single short block); `mma_read_end` is where the last stage's reads end, counted from
 * the 1 KB-aligned start of the ring, and a plan is only ever made when it stays within
 * `smem_avail` (the allocation past the ring start, with the worst-case alignment pad).
 */
typedef struct EngramProjectPlan {
  int32_t grid, threads, smem_bytes;  /* launch: CTAs (persistent, <= num_sms), threads, dynamic smem */
  int32_t tile_rows, tile_cols;       /* token rows x wkv rows per tile (128 or 256 x 16..256, or a split tile) */
  int32_t split;                      /* 2: two 128-row CTAs share a 2x-wide column block (bf16 only) */
  int32_t token_rows_loaded;          /* token rows the TMA loads per 128-row half (128, or fewer) */
  int32_t stages, stage_bytes;        /* ring depth and bytes per stage */
  int32_t tmem_cols;                  /* tensor-memory columns allocated */
  int32_t stream_k;                   /* 1: stream-K schedule */
  int32_t mma_read_end, smem_avail;   /* see above: mma_read_end <= smem_avail always */
} EngramProjectPlan;
int engram_project_plan(int64_t T, int32_t K, int32_t N, int32_t wkv_format, int32_t num_sms,
                        EngramProjectPlan* out);

/* Workspace bytes that let engram_project run the stream-K schedule for this shape on the current
 * device (0: the shape always runs the data-parallel schedule, or bad sizes). */
size_t engram_project_workspace_bytes(int64_t T, int32_t K, int32_t N);

/* Tuning knob for engram_project: force the tile width (columns per CTA, a multiple of 16 in
 * [16, 256]); 0 restores the automatic choice. A forced width also turns off the split tiles the
 * automatic choice uses for 129..256 tokens (pairs of 128-row CTAs on twice as many columns).
 * Process-wide; not thread-safe against calls. */
void engram_set_gemm_tile(int32_t bn);
/* Tuning knob for engram_project: 1 forces the data-parallel tile schedule, 2 the stream-K
 * schedule (when the workspace allows), 0 restores the automatic choice. Process-wide. */
void engram_set_gemm_schedule(int32_t s);

/*
 * FP8 operand variant of stage 3 (MXFP8). The FP8 table of [vLLM] ParallelEngramEmbedding
 * (float8_e4m3fn weight, one ue8m0 scale per 32 values) already is an MXFP8 operand; this
 * variant gathers its rows without dequantising them and multiplies them with a wkv stored the
 * same way on the tensor cores' block-scaled path (tcgen05.mma kind::mxf8f6f4), fp32 out. The
 * result equals the projection of the dequantised operands with fp32 accumulation. It needs no
 * workspace. Scale bytes are E8M0 exponents (value = code * 2^(byte - 127)).
 *
 * Scale layout (both operands): the bytes of a matrix with R rows and K columns are stored as
 * [ceil(K/128)][R4][4] with R4 = R rounded up to a multiple of 4: byte (kb, r, j) is the scale of
 * row r's block of 32 columns 4*kb + j. Each 128-column step of the projection then reads one
 * contiguous run per operand. Pad rows (r >= R) are ignored.
 */

/* wkv bf16 [N, K] -> MXFP8: codes uint8 [N, K] (e4m3) and scales uint8 [ceil(K/128)][N4][4]. Per row and
 * block of 32 along K, the scale is the smallest power of two 2^e with max|w| / 2^e <= 448 (byte
 * 127 + e; the table's own scale convention, so no value saturates) and each code is w / 2^e
 * rounded to the nearest e4m3 value, ties to even; an all-zero block gets byte 127 and zero codes.
 * K % 32 == 0; scales 4-byte aligned. Device pointers; deterministic. */
int engram_quantize_mxfp8(const uint16_t* w, int64_t N, int32_t K, uint8_t* codes, uint8_t* scales,
                          engram_stream_t stream);

/* Stage 2 for the FP8 variant: like engram_gather_dequant for an FP8_E8M0 table, but the rows'
 * codes and scale bytes are copied as they are: codes uint8 [T, C*head_dim], scales in the layout
 * above, uint8 [ceil(C*head_dim/128)][T4][4]. Ids outside [0, num_rows) give a zero row (codes 0,
 * scale byte 127) and set ENGRAM_ERR_ROW_ID. head_dim % 32 == 0; table, codes, scales 16-byte
 * aligned. */
int engram_gather_fp8_codes(const int32_t* ids, int64_t ids_stride_t, int64_t T, int32_t C,
                            int32_t head_dim, const void* table, const uint8_t* table_scales,
                            int64_t num_rows, uint8_t* codes, uint8_t* scales, int32_t* err_flag,
                            engram_stream_t stream);

/* Stage 3, FP8 variant: kv fp32 [T, N] = A * W^T with A codes [T, K] + A_scales [K/128][T4][4]
 * (from engram_gather_fp8_codes) and W codes [N, K] + W_scales [K/128][N4][4] (from
 * engram_quantize_mxfp8). K % 128 == 0, N % 16 == 0; all pointers 16-byte aligned. err_flag as
 * for engram_project. */
int engram_project_mxfp8(const uint8_t* A, const uint8_t* A_scales, const uint8_t* W,
                         const uint8_t* W_scales, float* kv, int64_t T, int32_t K, int32_t N,
                         int32_t* err_flag, engram_stream_t stream);

/* Tuning knob for engram_project_mxfp8: force the tile width (a multiple of 16 in [16, 256] that
 * fits tensor memory); 0 restores the automatic choice. Process-wide. */
void engram_set_gemm_mx_tile(int32_t bn);

/*
 * Stage 4: gate, in place on the fp32 highway ([NeMo] _engram_gate_core; [vLLM]
 * Engram.forward; [Atlas] stage 4). For each token t with token_mask[t] != 0 and stream j:
 *   s   = <h_j * rsqrt(mean(h_j^2)+eps) * q_weight[j], key_j * rsqrt(mean(key_j^2)+eps) * k_weight[j]> / sqrt(H)
 *   g   = sigmoid( sign(s) * sqrt(max(|s|, clamp)) )
 *   h_j = h_j + g * value
 * Masked tokens are not read or written.
 *   streams   device fp32 [T, hc, H] (in/out), 16-byte aligned
 *   kv        device fp32 [T, (hc+1)*H] (output of engram_project)
 *   q_weight, k_weight device bf16 [hc, H]
 *   token_mask device uint8 [T] or NULL
 *   err_flag  device int32 or NULL: ENGRAM_ERR_PIPE_TIMEOUT if a copy into shared memory never
 *             completed (the streams of the items not yet processed are then unchanged)
 * H % 8 == 0, 8 <= H <= 8192, 1 <= hc <= 8. A persistent kernel (a few CTAs per SM), each
 * CTA streaming its (token, stream) rows through shared memory with bulk copies.
 */
int engram_gate(const EngramDims* dims, float* streams, const float* kv,
                const uint16_t* q_weight, const uint16_t* k_weight, const uint8_t* token_mask,
                int64_t T, int32_t* err_flag, engram_stream_t stream);

/* Tuning knob for engram_gate (and the gate inside engram_forward): 1 forces the persistent kernel
 * (a few CTAs per SM streaming (token, stream) rows through shared memory), 2 the one-CTA-per-item
 * kernel (every load of a (token, stream) item in registers at once, for few items), 0 restores the
 * automatic choice (one CTA per item up to 8 items per SM). Process-wide; not thread-safe against
 * calls. Both give the same results up to fp32 summation order. */
void engram_set_gate_form(int32_t form);

/*
 * Tuning knob for engram_forward (and engram_forward2 / engram_forward_noalloc): how the gate
 * joins the projection ([NeMo] compile_engram_gate fuses the gate's reductions; [vLLM]
 * Engram.forward runs the gate right after the wkv projection). Same results as the separate
 * gate up to fp32 summation order; the projection then runs its data-parallel schedule.
 *   0  (the default) the gate is its own kernel after the projection.
 *   1  key reductions in the projection's epilogue: the key columns of kv are never stored; for
 *      every token row of a tile the epilogue forms, per stream the tile covers, sum key^2 and
 *      sum (h * q_weight) * (key * k_weight) from the stream row and the accumulators, and a
 *      finishing pass adds sum h^2, forms the gate and adds g * value. Layers with
 *      hidden % 32 == 0 whose projection tiles are at most `hidden` columns wide (others run
 *      mode 0).
 *   2  the gate inside the projection kernel, overlapped with it: eight more warps per CTA apply
 *      the gate to the tokens of each 128- or 256-row block as soon as every tile of that block
 *      is stored, while the tensor cores work on later tiles (bf16 wkv layers; others run mode 0).
 * Process-wide; not thread-safe against calls.
 */
void engram_set_gate_fusion(int32_t mode);

/*
 * Tuning knob for engram_forward (and engram_forward2 / engram_forward_noalloc): 1 lets the FP8
 * variant's projection gather its token rows from the table itself ([vLLM] _engram_lookup_kernel
 * stages the rows the wkv projection consumes; here they go straight into the projection's operand
 * tiles in shared memory, never through a gathered copy in HBM). The gathers before it then write
 * only the rows' scale words. Applies to layers with an MXFP8 wkv, head_dim % 128 == 0 and fewer
 * than 2^31 table rows. Same results as with the gathered copy (bit-identical kv). 0 (the default)
 * turns it off. Process-wide; not thread-safe against calls.
 */
void engram_set_operand_gather(int32_t on);

/*
 * Tuning knob for engram_forward (and engram_forward2 / engram_forward_noalloc): the order in which
 * a layer's gather reads the table ([vLLM] ParallelEngramEmbedding.lookup sorts a lookup's ids
 * before reading a table in host memory; _engram_lookup_thresholds). 0 (the default): token order,
 * the leading FP8 layers' rows fetched by the hash launch. 1: table order: per layer, the
 * (token, column) rows are grouped by table region (at most 16384 regions, by id >> shift) with a
 * counting pass, a scan and a scatter into a permutation (four more launches per layer, their
 * scratch in the workspace), then the gather walks the permutation and writes every row at its own
 * place. The results are bit-identical to token order. Process-wide; not thread-safe against calls.
 */
void engram_set_gather_order(int32_t mode);

/* Per-layer resident weights ([Atlas] EngramLayerWeights; [vLLM] Engram parameters). */
typedef struct EngramLayerWeights {
  int32_t table_format;        /* EngramTableFmt */
  const void* table;           /* device, see engram_gather_dequant */
  const uint8_t* table_scales; /* device, FP8_E8M0 only */
  int64_t table_rows;
  const uint16_t* wkv;         /* device [(hc+1)*H, C*head_dim]: bf16, or e4m3 codes (MXFP8) */
  const uint16_t* q_weight;    /* device bf16 [hc, H] */
  const uint16_t* k_weight;    /* device bf16 [hc, H] */
  int32_t wkv_format;          /* EngramWkvFmt; MXFP8 needs an FP8_E8M0 table and K % 128 == 0 */
  const uint8_t* wkv_scales;   /* device, MXFP8 only: [C*head_dim/128][N4][4] (see engram_project_mxfp8) */
} EngramLayerWeights;

/* Hash tables ([Atlas] EngramHashTables). All device memory. */
typedef struct EngramHashTables {
  const int32_t* token_map;   /* [raw_vocab] */
  const int64_t* multipliers; /* [layers, max_ngram] */
  const int64_t* primes;      /* [layers, C] */
  const int64_t* offsets;     /* [layers, C] */
} EngramHashTables;

/* One call's tokens. All device memory; see engram_hash. */
typedef struct EngramTokens {
  const int32_t* input_ids;
  int64_t T;
  const int32_t* cu_seqlens;
  int32_t num_seqs;
  const int32_t* sequence_ids;
  const uint8_t* token_mask;
  const int32_t* lookback_ids;
} EngramTokens;

/* Minimum bytes of device workspace engram_forward needs for T tokens (256-byte aligned pieces:
 * hash ids [T, layers, C] int32; one operand slot per layer, holding its rows [T, C*head_dim]
 * bf16, or with an MXFP8 wkv its row codes [T, C*head_dim] and then the scale words
 * [ceil(C*head_dim/128)][T4][4]; kv [T, (hc+1)*H] fp32). Workspace beyond the minimum is handed
 * to the projection: add engram_project_workspace_bytes(T, C*head_dim, (hc+1)*H) for its
 * stream-K schedule. */
size_t engram_forward_workspace_bytes(const EngramDims* dims, int64_t T);

/*
 * The whole path. Every layer's rows are gathered before the first projection, as [vLLM]
 * prepare_embeddings stages every layer's input before the decoder layers: one hash launch for
 * all layers, which also fetches the rows of the leading run of FP8+E8M0 layers (at most 8), then
 * one gather launch per run of consecutive remaining layers with the same table format and wkv
 * format (at most 8 each); then per layer project -> gate.
 *   layers     host array [dims->layers] of per-layer weights
 *   streams    host array [dims->layers] of device fp32 [T, hc, H] highways, updated in place
 *   workspace  device, >= engram_forward_workspace_bytes(dims, T), 256-byte aligned (see there
 *              for the optional extra that speeds up the projection)
 *   out_ids    device int32 [T, layers, C] or NULL: if given, the hash writes the ids there
 *              (and the workspace's id region goes unused)
 * Launches 1 + (gather launches) + 2*layers kernels on `stream`: 3 for one FP8 layer, 4 for one
 * Q2_K or bf16 layer, 6 for two layers of one format.
 */
int engram_forward(const EngramDims* dims, const EngramHashTables* tables,
                   const EngramLayerWeights* layers, const EngramTokens* tokens,
                   float* const* streams, void* workspace, size_t ws_bytes, int32_t* out_ids,
                   int32_t* err_flag, engram_stream_t stream);

/*
 * engram_forward with a second caller stream for the row gathers of the later layers ([vLLM]
 * Engram._start_prefetch / _ready_rows: the next engram layers' rows are staged on a side stream
 * while the current layer computes). The hash (with the leading FP8 layers' rows) and layer 0's
 * rows run on `stream`; the gathers of the other layers run on side_stream once the hash is done,
 * and each layer's projection on `stream` waits for its rows. The ordering uses CUDA events the
 * library creates once per device (no device memory, no device-side waits); a call's records and
 * waits are enqueued under a lock, so calls from several host threads stay correct. Every piece of
 * work the call puts on side_stream is waited for by `stream` before its last projection, so work
 * ordered after the call on `stream` alone sees all of it.
 *   side_stream  a cudaStream_t; NULL or equal to `stream`: exactly engram_forward.
 * Other arguments and results as engram_forward (bit-identical streams).
 */
int engram_forward2(const EngramDims* dims, const EngramHashTables* tables,
                    const EngramLayerWeights* layers, const EngramTokens* tokens,
                    float* const* streams, void* workspace, size_t ws_bytes, int32_t* out_ids,
                    int32_t* err_flag, engram_stream_t stream, engram_stream_t side_stream);

/* Size of the static device scratch of engram_forward_noalloc: 32 MiB, held by every GPU that
 * loads the library until the process exits. */
#define ENGRAM_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * engram_forward without a workspace argument, for callers that may not allocate device memory:
 * e.g. an engine whose pool owns all the device memory it may touch and lends a plugin only its
 * own tensors, or a real-time loop that cannot take cudaMalloc's implicit synchronisation.
 * No page counterpart: the pages have no such entry point; the path computed is engram_forward's.
 *   Arguments as engram_forward, minus workspace/ws_bytes. The hash ids, rows and kv live in one
 *   static device array of ENGRAM_NOALLOC_SCRATCH_BYTES; a call whose
 *   engram_forward_workspace_bytes(dims, T) exceeds it returns ENGRAM_EINVAL and launches nothing
 *   (the decode step of 256 tokens, 24 hash columns of 256, hidden 4096, hc 4 needs 24.1 MB).
 *   The first call on each device looks up the array's device address (cudaGetSymbolAddress, with
 *   that device current): make that first call before any stream capture.
 *   Calls allocate nothing (no cudaMalloc, cudaFree or allocating library routine). All calls share
 *   the array and it keeps the last call's contents; nothing in it needs to start at zero. Calls
 *   whose work overlaps on the GPU (other streams or threads) race on it: order them.
 */
int engram_forward_noalloc(const EngramDims* dims, const EngramHashTables* tables,
                           const EngramLayerWeights* layers, const EngramTokens* tokens,
                           float* const* streams, int32_t* out_ids, int32_t* err_flag,
                           engram_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_H_ */
