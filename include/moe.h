/*
 * moe.h -- C ABI of libmoe_gb300.so: the MoE expert-FFN forward on one
 * GB300 (sm_103a).
 *
 *   align -> gather + grouped GEMM(w13) + SiLU(gate)*up
 *         -> grouped GEMM(w2) x routing weight -> combine
 *
 * The operation is the one the header comment of "factor_moe_fused_gemm.cu"
 * (ex_engine, Factor 2: MOE_FUSED_GEMM) spells out as its "Current PyTorch
 * path": per expert, gather the routed token rows, gate_up = x W13[e]^T,
 * act = SiLU(gate) * up, y = act W2[e]^T, and index-add weight * y back
 * into the token rows.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library allocates nothing and frees nothing; intermediates live in a
 *    caller-provided workspace (moe_workspace_size).
 *  - Tensors are dense, row-major, without padding between rows.
 *  - `stream` is a cudaStream_t passed as void*; every call is asynchronous
 *    on that stream and never synchronises the host, except
 *    moe_get_device_status, which does.
 *  - Argument and shape errors are detected on the host before any launch
 *    and returned as a status; nothing is launched then.  Launch failures
 *    return MOE_ERR_CUDA.  Errors found by the kernels themselves (an expert
 *    id outside [0, E), a pipeline wait that ran out) are written to a
 *    device status word (one int32 in device memory, 0 = no error, the first
 *    error wins); kernels that find it non-zero at start return without
 *    writing their outputs.  Read it with moe_get_device_status.
 *  - Expert ids are int32 in [0, E); routing weights are fp32.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum      */
    MOE_ERR_UNSUPPORTED = 2,   /* shape/dtype combination this build lacks   */
    MOE_ERR_WORKSPACE = 3,     /* workspace too small or misaligned          */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed          */
    MOE_ERR_DEVICE_BAD_ID = 5, /* (device) an expert id outside [0, E)       */
    MOE_ERR_TIMEOUT = 6,       /* (device) a pipeline wait ran out; the      */
                               /* kernel stopped, freed its tensor memory    */
                               /* and returned                               */
    MOE_ERR_BOUNDS = 7         /* (device, checked build only) an index read */
                               /* from an input or the workspace lay outside */
                               /* the buffer it addresses; the access was    */
                               /* skipped                                    */
} moe_status_t;

typedef enum {
    MOE_F32 = 0,     /* IEEE binary32                                          */
    MOE_BF16 = 1,    /* bfloat16                                               */
    MOE_E4M3 = 2,    /* OCP FP8 E4M3 (finite-only variant)                     */
    MOE_E2M1_MX = 3  /* OCP MX FP4: e2m1 pairs, lower K index in the low       */
                     /* nibble, plus one e8m0 scale byte per 32 K elements     */
} moe_dtype_t;

/* Activation of the first GEMM's epilogue (moe_problem_t.activation). */
typedef enum { MOE_ACT_SILU = 0, MOE_ACT_SWIGLU_CLAMP = 1 } moe_activation_t;

/* One MoE layer.  T tokens of width H, E experts with intermediate size I,
 * top-K routing.
 *   act    : dtype of x and out: MOE_F32 or MOE_BF16.
 *   weight : dtype of w13/w2: equal to act, or MOE_E2M1_MX (then act must
 *            be MOE_BF16; x is cast to e4m3 with one fp32 scale per row and
 *            the hidden activation is stored as e4m3(a / h_scale)).
 *   block_m: rows per alignment block (16, 32, 64, 128 or 256; MX weights:
 *            128), 0 = automatic: 256 when bf16/fp32 experts receive at
 *            least 256 rows on average (T*K >= 256*E), else 128.  The
 *            bf16/fp32 GEMMs take one block as the N side of a tile and
 *            spend MMA work only on its valid rows (rounded up to 16).
 *   h_scale: scale of the e4m3 hidden activation (MX weights only; 0 => 1).
 *   expert_base, local_experts: expert-parallel shard (local_experts = 0:
 *            no sharding).  The layer's experts [expert_base,
 *            expert_base + local_experts) live here; w13/w2 (and their
 *            scales) hold those experts only, indexed from 0.  Ids still
 *            range over [0, E); a slot routed to another shard's expert
 *            contributes nothing, so out is this shard's share of the layer
 *            output and the shards' outputs sum to the unsharded one.
 *            Source: "MOE Bmm1 Fused Gather", init_routing_data (a shard
 *            keeps the histogram of its local experts; experts split into
 *            equal contiguous ranges by make_expt_dict_uniform).
 *   activation, swiglu_alpha, swiglu_limit, gate_up_interleaved, w13_bias,
 *   w2_bias: the expert FFN's activation and biases (L = experts held).
 *            MOE_ACT_SILU: a = SiLU(g) * u, the plain SwiGLU of
 *            "factor_moe_fused_gemm.cu".  MOE_ACT_SWIGLU_CLAMP: GPT-OSS's
 *            variant from "MOE Bmm1 Fused Gather" (_swiglu_step1/2): g =
 *            min(g, limit), u = clamp(u, -limit, limit),
 *            a = g * sigmoid(alpha * g) * (u + 1).  g and u are the
 *            accumulators plus w13_bias (per expert and w13 row, that page's
 *            apply_bias_and_scale); y = W2 a + w2_bias before the routing
 *            weight.  Either bias may be NULL (zero) and goes with either
 *            activation.  gate_up_interleaved: w13 (and w13_bias) hold gate
 *            and up in alternating rows, that page's layout, instead of the
 *            two halves; for MX weights pass the same flag to
 *            moe_pack_mx_weights, whose packed form is always in halves.
 *   fused_combine: 0 = the deterministic combine: GEMM2 writes each weighted
 *            expert row in sorted order and moe_combine sums every token's K
 *            rows in k order.  1 = the combine fused into GEMM2, after the
 *            scatter-add of "factor_moe_fused_gemm.cu"
 *            (weighted_scatter_add_kernel): GEMM2's epilogue adds each
 *            weighted row into an fp32 (T, H) accumulator with atomic adds
 *            (zeroed by the gather step before) and moe_combine_finish
 *            rounds it to out.  The order of the adds is not fixed, so the
 *            fp32 sums, and rarely the rounded outputs, may differ between
 *            runs in the last bits.  The workspace then holds T*H fp32
 *            instead of k_splits*cap*H. */
typedef struct {
    int T, H, I, E, K;
    int act;
    int weight;
    int block_m;
    float h_scale;
    int expert_base;
    int local_experts;
    int activation;           /* moe_activation_t                          */
    float swiglu_alpha;       /* MOE_ACT_SWIGLU_CLAMP: sigmoid slope       */
    float swiglu_limit;       /* MOE_ACT_SWIGLU_CLAMP: clamp, > 0          */
    int gate_up_interleaved;  /* w13 rows 2j = gate j, 2j+1 = up j         */
    const float* w13_bias;    /* device (L, 2I) fp32 in w13's row order    */
    const float* w2_bias;     /* device (L, H) fp32                        */
    int fused_combine;        /* 0 or 1, see above                         */
} moe_problem_t;

/* Sub-buffers of the moe_forward workspace (byte offsets, see
 * moe_workspace_offsets). */
typedef enum {
    MOE_WS_STATUS = 0,         /* int32 device status word                  */
    MOE_WS_COUNTS = 1,         /* int32[L]   (L = local experts, E unsharded) */
    MOE_WS_OFFSETS = 2,        /* int32[L+1]                                */
    MOE_WS_PADDED_OFFSETS = 3, /* int32[L+1]                                */
    MOE_WS_SORTED_IDS = 4,     /* int32[cap]                                */
    MOE_WS_INV_PERM = 5,       /* int32[T*K]                                */
    MOE_WS_BLOCK_INFO = 6,     /* int32[cap/block_m][4]                     */
    MOE_WS_NUM_BLOCKS = 7,     /* int32[1]                                  */
    MOE_WS_XQ = 8,             /* A rows in sorted order [cap][H]: e4m3     */
                               /* (MX weights) or act rows                  */
    MOE_WS_X_SCALE = 9,        /* fp32[T]      (MX weights only)            */
    MOE_WS_H = 10,             /* act or e4m3 [cap][I]                      */
    MOE_WS_Y = 11,             /* fp32[splits][cap][H], or fp32[T][H] when  */
                               /* fused_combine (the accumulator)           */
    MOE_WS_ALIGN = 12,         /* int32 per-warp counts of the align of     */
                               /* large batches (T*K >= 16384), else empty  */
    MOE_WS_NUM = 13
} moe_ws_part_t;

/* Static string for a status code (never NULL). */
const char* moe_status_string(int status);

/* Library ABI version (increments on any signature change). */
int moe_abi_version(void);

/* Rows per alignment block the GEMMs of this build use for `p` (resolves
 * block_m == 0), or -1 when p is invalid. */
int moe_resolve_block_m(const moe_problem_t* p);

/* Capacity of the padded sorted list: T*K + min(E, T*K)*(block_m - 1).
 * Every active expert's list is padded to a multiple of block_m, so this
 * bounds sum_e ceil(count_e / block_m) * block_m for any routing. */
size_t moe_align_capacity(int T, int K, int E, int block_m);

/* Number of K splits moe_forward uses for the down projection of `p`
 * (its fp32 partial outputs are summed by the combine). */
int moe_gemm2_default_splits(const moe_problem_t* p);

/* Bytes of workspace moe_forward needs for `p` (0 when p is invalid). */
size_t moe_workspace_size(const moe_problem_t* p);

/* Byte offset of every moe_ws_part_t inside the workspace, written to
 * offsets[MOE_WS_NUM].  Parts a problem does not use get size 0. */
int moe_workspace_offsets(const moe_problem_t* p, size_t offsets[MOE_WS_NUM],
                          size_t sizes[MOE_WS_NUM]);

/* ---- align ------------------------------------------------------------
 * Source: "factor_moe_fused_gemm.cu", build_expert_map_kernel (expert
 * histogram, CSR offsets, permutation) and "moe triton kernel use tma"
 * (LightLLM pull request 1100), the summary's mblocks_to_tuple_info
 * (expert id, M-index and token start of each M-block).
 *
 * With i = t*K + k the flat index of token t's k-th choice (N_a = T*K):
 *   counts[e]                 number of i with topk_ids[i] == e      int32[E]
 *   offsets[e]                exclusive prefix sum of counts         int32[E+1]
 *   padded_offsets[e]         exclusive prefix sum of
 *                             ceil(counts/block_m)*block_m           int32[E+1]
 *   sorted_ids[s]             slot s of the padded expert-sorted list: the
 *                             r-th smallest i routed to e sits at
 *                             padded_offsets[e] + r (stable order);
 *                             every other slot < cap holds N_a       int32[cap]
 *   inv_perm[i]               the slot of i                          int32[N_a]
 *   block_info[b]             {expert, m, first slot, valid rows} of block
 *                             b < num_blocks (experts ascending);
 *                             {-1, 0, 0, 0} for the rest    int32[cap/block_m][4]
 *   num_blocks[0]             padded_offsets[E] / block_m            int32[1]
 * cap = moe_align_capacity(T, K, E, block_m); block_m in {16,32,64,128}.
 * E <= 1024.  An id outside [0, E) makes the kernel write num_blocks = 0,
 * set MOE_ERR_DEVICE_BAD_ID in *dev_status (when dev_status is not NULL)
 * and leave the other outputs unspecified.  T == 0 writes nothing and
 * returns MOE_OK. */
int moe_align(const int32_t* topk_ids, int T, int K, int E, int block_m, int32_t* counts,
              int32_t* offsets, int32_t* padded_offsets, int32_t* sorted_ids, int32_t* inv_perm,
              int32_t* block_info, int32_t* num_blocks, int32_t* dev_status, void* stream);

/* moe_align for one expert-parallel shard holding experts
 * [expert_base, expert_base + local_experts) of E.  Every per-expert output
 * (counts, offsets, padded_offsets, the expert field of block_info) covers
 * the local experts only, indexed e - expert_base; assignments to other
 * experts are left out of the lists and get inv_perm[i] = -1.  cap =
 * moe_align_capacity(T, K, local_experts, block_m).  Ids are still checked
 * against [0, E).  expert_base = 0, local_experts = E is moe_align.
 * Source: "MOE Bmm1 Fused Gather", init_routing_data (the local experts'
 * histogram of one shard).  1 <= local_experts <= 1024,
 * expert_base + local_experts <= E, else MOE_ERR_INVALID_ARG /
 * MOE_ERR_UNSUPPORTED.
 * scratch / scratch_bytes: device memory of at least
 * moe_align_scratch_bytes(T, K, local_experts) bytes (16-byte aligned, may
 * be NULL when that is 0 or to keep one CTA).  With it, batches of 16384 or
 * more assignments are aligned by many CTAs (per-warp histograms in the
 * scratch, one scan CTA, a scatter over many CTAs) -- the same outputs,
 * as moe_forward does; without it, by one CTA. */
int moe_align_local(const int32_t* topk_ids, int T, int K, int E, int expert_base,
                    int local_experts, int block_m, int32_t* counts, int32_t* offsets,
                    int32_t* padded_offsets, int32_t* sorted_ids, int32_t* inv_perm,
                    int32_t* block_info, int32_t* num_blocks, void* scratch,
                    size_t scratch_bytes, int32_t* dev_status, void* stream);

/* Scratch bytes moe_align_local uses for T*K assignments over
 * local_experts experts: 0 below 16384 assignments. */
size_t moe_align_scratch_bytes(int T, int K, int local_experts);

/* ---- routing + align ------------------------------------------------------
 * The router step before the path, folded into align.  Source: "MOE Bmm1
 * Fused Gather", init_routing_data: topk(logits, k, apply_softmax) over the
 * router logits, whose expert histogram feeds the ragged metadata.
 *   logits        (T, E) logit_dtype (MOE_F32 or MOE_BF16), row-major
 *   topk_ids      (T, K) int32 out: the experts of the K largest logits of
 *                 each token in descending order, an equal logit going to
 *                 the lower expert id (compared at the logits' own values)
 *   topk_weights  (T, K) fp32 out: softmax over the E experts renormalised
 *                 over the K chosen = softmax over the K chosen logits
 * then moe_align_local over those ids (all other outputs as there).  Up to
 * 1024 tokens the align kernel routes the batch itself (one launch); larger
 * batches are routed by a kernel of a warp per token first.  K <= 32,
 * E <= 1024.  A token whose logits are NaN where a choice is made records
 * MOE_ERR_DEVICE_BAD_ID. */
int moe_route_align(const void* logits, int logit_dtype, int T, int E, int K, int expert_base,
                    int local_experts, int block_m, int32_t* topk_ids, float* topk_weights,
                    int32_t* counts, int32_t* offsets, int32_t* padded_offsets,
                    int32_t* sorted_ids, int32_t* inv_perm, int32_t* block_info,
                    int32_t* num_blocks, int32_t* dev_status, void* stream);

/* ---- mxfp4 weight packing (once, when the model is loaded) -----------------
 * Source: "MOE Bmm1 Fused Gather" -- its matmul takes the e2m1 weights in a
 * pre-shuffled value layout and the e8m0 scales in a swizzled scale layout,
 * both made for its kernel's tiles before the kernel runs.  This library's
 * block-scaled GEMMs likewise read MX weights in a packed form:
 *   natural form of a weight tensor with E experts, R rows, K elements along
 *   the reduction: values (E, R, K/2) bytes, e2m1 pairs, lower K index in the
 *   low nibble; scales (E, R, K/32) e8m0 bytes.
 *   The R rows of an expert form `sections` equal sections (2 for w13: gate
 *   rows and up rows; 1 for w2); K is cut into Kp/128 tiles of 128 elements
 *   (Kp = K rounded up to 128).
 *   packed values: tile-major (E, NT, Kp/128, 192, 64) bytes (NT as for the
 *   scale images below): byte 64*r + b of tile (e, n, t) holds natural bytes
 *   64*t + b (K elements 128*t + 2b, 2b + 1) of row r of weight tile n (the
 *   same tile rows as the scale images), zero nibbles past K or past the
 *   section's rows.  One tile is 12 KB of consecutive bytes, which one TMA
 *   copy expands into the 16-byte slots the MMA reads 4-bit operands from.
 *   packed scales: 1 KB images (E, NT, Kp/128, 1024), one per 192-row
 *   weight tile n and K tile t: NT = ceil((R/2)/96) tiles of 96 rows of
 *   each section (w13: tile row r < 96 is gate row 96n + r, r >= 96 is up
 *   row 96n + r - 96), or NT = ceil(R/192) tiles of 192 rows (w2: tile row
 *   r is row 192n + r).  Byte 512*p + 16*l + 4*c + b of image (e, n, t) is
 *   the scale of tile row 128*p + 32*c + l, K block 4*t + b, and 127 where
 *   that row or block does not exist -- the layout tensor memory takes the
 *   scales in.
 * moe_mx_packed_bytes returns the total bytes (0 on bad arguments) and the
 * two parts; K must be a multiple of 32.  moe_pack_mx_weights writes the
 * packed form on `stream` (all pointers device memory; the packed values
 * must be 32-byte and the images 16-byte aligned to be used).  interleaved
 * = 1 (sections = 2 only): the natural rows hold the two sections
 * alternately (row 2j of section 0, row 2j+1 of section 1, GPT-OSS's gate /
 * linear layout); the packed form is the same as for the halves. */
size_t moe_mx_packed_bytes(int E, int R, int K, int sections, size_t* value_bytes,
                           size_t* scale_bytes);
int moe_pack_mx_weights(const uint8_t* w, const uint8_t* w_scale, int E, int R, int K,
                        int sections, int interleaved, uint8_t* w_packed, uint8_t* scale_packed,
                        void* stream);

/* ---- fp8 activation step ------------------------------------------------
 * Source: "MOE Bmm1 Fused Gather" (Triton Gluon example), pack_e4m3x2
 * (fp32 -> e4m3, round to nearest even, saturating).  Reading: one scale
 * per row, s_t = amax_t / 448 (1 when the row is zero), both formed in fp32.
 *   x         (T, H) in x_dtype (MOE_BF16 or MOE_F32)
 *   xq        (T, H) e4m3 codes, = e4m3_rn_satfinite(x / s_t)
 *   row_scale (T) fp32 s_t                                                  */
int moe_quantize_x_fp8(const void* x, int x_dtype, int T, int H, uint8_t* xq, float* row_scale,
                       void* stream);

/* The same step with the token gather fused in, for the block-scaled GEMMs:
 * each token's codes are written to every slot of the expert-sorted list the
 * token occupies, xq_sorted[inv_perm[t*K + k], :] (cap rows of H bytes; rows
 * of padding slots are not written), scales as above in token order.
 * inv_perm as written by moe_align.  acc_zero: NULL, or the fp32 (T, H)
 * accumulator of a fused combine, whose rows this step sets to zero.
 * Skipped when *dev_status != 0. */
int moe_quantize_gather_x_fp8(const void* x, int x_dtype, int T, int H, int K,
                              const int32_t* inv_perm, uint8_t* xq_sorted, float* row_scale,
                              float* acc_zero, int32_t* dev_status, void* stream);

/* ---- gather step (bf16/fp32 weights) ---------------------------------------
 * Source: "MOE Bmm1 Fused Gather", load_activations (token rows gathered by
 * index), done as its own pass.
 * Token rows to sorted slots: x_sorted[inv_perm[t*K + k], :] = x[t, :] for
 * every choice of every token (rows of padding slots are not written; a
 * negative inv_perm entry, another shard's slot, is skipped); x (T, H) in
 * dtype (MOE_BF16 / MOE_F32), x_sorted (cap, H), inv_perm from moe_align.
 * The bf16/fp32 gate/up GEMM reads its token rows in this sorted form.
 * acc_zero: NULL, or the fp32 (T, H) accumulator of a fused combine, whose
 * rows this step sets to zero (H a multiple of 4).
 * Skipped when *dev_status != 0. */
int moe_gather_rows(const void* x, int dtype, int T, int H, int K, const int32_t* inv_perm,
                    void* x_sorted, float* acc_zero, int32_t* dev_status, void* stream);

/* ---- gather + GEMM1 + SiLU*up -------------------------------------------
 * Source: "factor_moe_fused_gemm.cu", fused_silu_gate_kernel (gate = first
 * half of the w13 rows, up = second half, SiLU(g) = g / (1 + e^-g)) and
 * "MOE Bmm1 Fused Gather", load_activations (token rows gathered by index,
 * padded rows masked) with epilogue_partition (activation fused into the
 * GEMM epilogue).
 * For every slot s of a block b < *num_blocks with i = sorted_ids[s] < N_a
 * and e = block_info[b].expert:
 *   h[s, j] = SiLU(W13[e, j, :] . x[i / K, :]) * (W13[e, I + j, :] . x[i / K, :])
 * x    the token rows in sorted order (cap, H): act rows as written by
 *      moe_gather_rows, or for MX weights the e4m3 codes as written by
 *      moe_quantize_gather_x_fp8, with x_row_scale (T) fp32
 * w13  (E, 2I, H) weight dtype (MX: packed values + scale images of
 *      moe_pack_mx_weights with R = 2I, K = H, sections = 2)
 * h    (cap, I) act (MX: e4m3 codes of a / h_scale); rows of padding slots
 *      are not written.  H and I must be multiples of 64 (32 for MOE_F32 and
 *      for MX weights).
 * sorted_ids/block_info/num_blocks as written by moe_align with the same
 * block_m (MX weights: 128).  dev_status may be NULL. */
int moe_gemm1_silu(const moe_problem_t* p, const void* x, const float* x_row_scale,
                   const void* w13, const uint8_t* w13_scale, const int32_t* sorted_ids,
                   const int32_t* block_info, const int32_t* num_blocks, void* h,
                   int32_t* dev_status, void* stream);

/* moe_gemm1_silu with the gather inside the GEMM ("MOE Bmm1 Fused Gather",
 * load_activations: the producer loads the token rows of a tile by index
 * into its shared-memory ring).  x is the (T, H) act tensor in token order;
 * the row of slot s is x[sorted_ids[s] / K], fetched four rows per TMA copy
 * (tile::gather4).  h is the same as moe_gemm1_silu writes from
 * moe_gather_rows' output, bit for bit.  bf16 / fp32 activations only: MX
 * weights return MOE_ERR_UNSUPPORTED (their fp8 step,
 * moe_quantize_gather_x_fp8, already gathers).  Other arguments, shapes and
 * errors as moe_gemm1_silu.  moe_forward keeps the separate gather pass:
 * a 4-row gather copy costs the producer far more than a tile box
 * (measured: even, within noise, at one token; slower from eight on). */
int moe_gemm1_silu_gather(const moe_problem_t* p, const void* x, const void* w13,
                          const int32_t* sorted_ids, const int32_t* block_info,
                          const int32_t* num_blocks, void* h, int32_t* dev_status,
                          void* stream);


/* ---- GEMM2 x routing weight -----------------------------------------------
 * Source: "moe triton kernel use tma", the review comment on
 * TOKEN_INPUT_USE_TMA (token rows of the down projection are contiguous in
 * sorted order and load as plain tiles; MUL_ROUTED_WEIGHT multiplies the
 * routing weight there) and the "Current PyTorch path"'s expert_out * weights.
 * For every valid slot s (as above) and split q < k_splits:
 *   y[q, s, c] = topk_weights[i] * sum_{j in split q} W2[e, c, j] * h[s, j]
 * so that sum_q y[q, s, :] is the routing-weighted expert output.  Splits
 * cut I into k_splits nearly equal runs of 64 columns (k_splits <= I/64).
 * h (cap, I) as written by moe_gemm1_silu; w2 (E, H, I) weight dtype (MX:
 * packed by moe_pack_mx_weights with R = H, K = I, sections = 1);
 * y (k_splits, cap, H) fp32, padding rows not written.  MX splits cut the
 * 128-element K tiles.
 * With p->fused_combine, y is instead the fp32 (T, H) accumulator, zeroed
 * beforehand (moe_gather_rows / moe_quantize_gather_x_fp8 with acc_zero),
 * and every split of every valid slot s adds its part of
 * topk_weights[i] * (W2[e] h[s] + b2) into row i / K with atomic adds. */
int moe_gemm2_weighted(const moe_problem_t* p, const void* h, const void* w2,
                       const uint8_t* w2_scale, const float* topk_weights,
                       const int32_t* sorted_ids, const int32_t* block_info,
                       const int32_t* num_blocks, float* y, int k_splits, int32_t* dev_status,
                       void* stream);

/* ---- combine ---------------------------------------------------------------
 * Source: the index_add of the "Current PyTorch path" and
 * weighted_scatter_add_kernel of "factor_moe_fused_gemm.cu", done here as a
 * deterministic per-token reduction instead of atomics:
 *   out[t, c] = sum_{k < K} sum_{q < k_splits} y[q, inv_perm[t*K + k], c]
 * summed in fp32 in k order, rounded once to out_dtype (MOE_F32/MOE_BF16);
 * a negative inv_perm entry (another shard's slot) adds nothing.
 * y (k_splits, cap, H) fp32; inv_perm (T*K); out (T, H). */
int moe_combine(const float* y, int k_splits, size_t cap, const int32_t* inv_perm, int T, int K,
                int H, int out_dtype, void* out, int32_t* dev_status, void* stream);

/* The last step of a fused combine (moe_problem_t.fused_combine):
 * out[t, c] = acc[t, c] rounded once to out_dtype (MOE_F32 / MOE_BF16).
 * acc (T, H) fp32 as GEMM2 left it; H a multiple of 4.  Skipped when
 * *dev_status != 0. */
int moe_combine_finish(const float* acc, int T, int H, int out_dtype, void* out,
                       int32_t* dev_status, void* stream);

/* ---- the whole forward -----------------------------------------------------
 * Runs align -> [fp8 step with the gather (MX) | gather] -> GEMM1 -> GEMM2
 * -> combine (with p->fused_combine: GEMM2 adding into the accumulator the
 * gather step zeroed -> moe_combine_finish) on `stream`; every
 * intermediate lives in `workspace` (device memory of at
 * least moe_workspace_size(p) bytes, 256-byte aligned, owned by the caller,
 * reusable across calls but not shared by calls in flight at once).
 *   x (T, H) act; topk_ids (T, K) int32; topk_weights (T, K) fp32;
 *   w13 (E, 2I, H), w2 (E, H, I) (MX: packed values and scale images of
 *   moe_pack_mx_weights); out (T, H) act.
 * The status word at MOE_WS_STATUS is cleared at the start of each call. */
int moe_forward(const moe_problem_t* p, const void* x, const int32_t* topk_ids,
                const float* topk_weights, const void* w13, const uint8_t* w13_scale,
                const void* w2, const uint8_t* w2_scale, void* out, void* workspace,
                size_t workspace_bytes, void* stream);

/* ---- the whole forward without a caller workspace ---------------------------
 * No counterpart on the pages: an addition of this library for callers that
 * cannot allocate device memory where they run the layer (a host framework
 * that owns and pre-carves all device memory, a serving loop that must not
 * allocate after start-up, a caller with no room to keep a workspace).
 * Same arguments and result as moe_forward, minus the workspace: the
 * intermediates go to one static device array of MOE_STATIC_SCRATCH_BYTES
 * inside the library, held on every GPU that loads it until the process
 * exits.  Allocates nothing (no cudaMalloc, no allocating library call).
 *  - Problems whose moe_workspace_size exceeds MOE_STATIC_SCRATCH_BYTES are
 *    rejected with MOE_ERR_WORKSPACE before anything is launched.
 *  - The first call on a device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - All calls on a device share the array, which keeps the last call's
 *    contents; the status word that must start at zero is cleared by each
 *    call.  Calls whose execution overlaps on the GPU race on the array:
 *    issue them in one stream order.
 *  - Argument errors give the same status codes as moe_forward.
 * Errors the kernels find (an expert id outside [0, E), a pipeline wait
 * that ran out) go to the device status word at offset 0 of the array, as
 * they do to a workspace's: the call still returns MOE_OK, later stages skip
 * their writes and out is left unspecified.  Read the word with
 * moe_forward_noalloc_status. */
#define MOE_STATIC_SCRATCH_BYTES (64u << 20)
int moe_forward_noalloc(const moe_problem_t* p, const void* x, const int32_t* topk_ids,
                        const float* topk_weights, const void* w13, const uint8_t* w13_scale,
                        const void* w2, const uint8_t* w2_scale, void* out, void* stream);

/* The device status word of the last moe_forward_noalloc on the current
 * device: synchronises `stream` and returns MOE_OK when the word is 0, its
 * code otherwise (as moe_get_device_status does for a workspace), or
 * MOE_ERR_CUDA.  No counterpart on the pages.  Allocates nothing. */
int moe_forward_noalloc_status(void* stream);

/* ---- test of the kernels' failure path (not for use in a model) -----------
 * Runs moe_gemm1_silu (gemm = 1) or moe_gemm2_weighted (gemm = 2) with the
 * same arguments (a_rows: x rows / hq codes for gemm 1, h for gemm 2; w and
 * w_scale: w13 or w2; k_splits: gemm 2 only), except that the kernel's
 * producers issue no copies at all and every pipeline wait gives up after
 * wait_limit_ns (1 ms to 2 s) of wall clock.  With nothing in flight the
 * first wait of each CTA runs out: the kernel raises its abort flag, frees
 * its tensor memory, writes MOE_ERR_TIMEOUT to *dev_status (which must not
 * be NULL to observe it) and returns; `out` is not written.  No counterpart
 * on the pages: it exists so that tests can drive the bounded waits
 * (MOE_ERR_TIMEOUT) without ever hanging a GPU. */
int moe_test_gemm_wait_timeout(const moe_problem_t* p, int gemm, const void* a_rows,
                               const float* x_row_scale, const void* w, const uint8_t* w_scale,
                               const float* topk_weights, const int32_t* sorted_ids,
                               const int32_t* block_info, const int32_t* num_blocks, void* out,
                               int k_splits, unsigned long long wait_limit_ns,
                               int32_t* dev_status, void* stream);

/* Launch geometry of the current device: its SM count and how many CTA pairs
 * of the bf16 gate/up kernel it holds at once (0 if unknown). */
int moe_device_info(int* sm_count, int* pair_clusters);

/* Synchronise `stream` and return the device status word at dev_status
 * (MOE_OK when it is 0), or MOE_ERR_CUDA if the stream itself failed. */
int moe_get_device_status(const int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
