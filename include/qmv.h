/*
 * qmv.h -- C ABI of libqmv: block-quantized decode matrix-vector products on
 * NVIDIA GB300 (sm_103a), dense and MoE expert-gathered.
 *
 * Operation. For a weight matrix W (N rows x K columns) stored block-quantized
 * and 1..16 decode (or speculative-verify) tokens, y = W . x per token.
 * Weight formats:
 *
 *   QMV_MXFP4  E2M1 4-bit codes, one E8M0 scale per 32 weights along K,
 *              times bf16 activations, fp32 accumulation, bf16 output.
 *              Source: "perf(rocm): add an mxfp4 arm to the warp-shared
 *              gather_qmv kernel for gpt-oss decode" (mlxcel #2178),
 *              "Current Behavior" and "Proposed Solution" item 1.
 *   QMV_MXFP8  E4M3 8-bit codes (OCP MX: exponent bias 7, subnormals,
 *              S.1111.111 = NaN, no infinity), one E8M0 scale per 32 weights,
 *              otherwise as MXFP4. The page lists the f16 MXFP4 and the
 *              MXFP8 gathers as the next scope beyond the bf16 MXFP4 arm
 *              (mlxcel #2178, "Scope").
 *   QMV_CB2    2-bit codes into a 4-entry int8 codebook, E8M0 per 16 weights.
 *   QMV_CB3    3-bit codes into an 8-entry int8 codebook, E8M0 per 16 weights.
 *   QMV_CB4    4-bit codes into a 16-entry int8 codebook, E8M0 per 32 weights.
 *              The codebook formats multiply q8_1 activations (int8 blocks of
 *              32 with an fp16 scale d) and reduce with integer dot products:
 *              y = sum_b d_b * sum_{h in b} 2^(e_h - 127) * sum_{i in h} lut[c_i] * q_i.
 *              Source: "perf(ggml/hip): optimize ROCMFPX fp3/fp2 MMVQ on RDNA
 *              (perm-LUT + VDR=4 + fp2)" (lucebox-hub #21), "Changes" and
 *              the review reply's "dot structure"; "DS4 H200: rocmfp2_mix MoE
 *              matvec 3.31x + ROCmFP4 dense matvec 1.53x" (geo-lucebox #31),
 *              "Headline" and "Caveats" (quantize_q8_1).
 *
 * E8M0 scale byte e means 2^(e-127); e = 255 means NaN.
 *
 * Conventions for every entry point:
 *  - Return 0 (QMV_OK) on success or a negative QMV_E* code. The message of
 *    the last failure on the calling thread is returned by qmv_last_error().
 *  - "_dev" pointers are CUDA device pointers owned by the caller; "_host"
 *    pointers are host memory owned by the caller. The library allocates no
 *    device memory and keeps no per-call state.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). GPU entry
 *    points only enqueue work: they never synchronize and never read device
 *    memory on the host. Argument errors are reported before anything is
 *    enqueued; launch errors come back as QMV_ECUDA.
 *  - Device pointers must be 16-byte aligned (QMV_EALIGN otherwise).
 *  - Invalid data on the device is not an error: an expert id outside
 *    [0, n_experts) yields a zero output row block; E8M0 = 255 yields NaN.
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QMV_OK 0
#define QMV_EINVAL (-1)  /* null pointer, bad format, ntok/top_k out of range */
#define QMV_ESHAPE (-2)  /* K % 32 != 0, N or K out of range, too many activation vectors */
#define QMV_EALIGN (-3)  /* a device pointer that is not 16-byte aligned */
#define QMV_ESIZE (-4)   /* a caller buffer smaller than the required size */
#define QMV_ECUDA (-5)   /* a CUDA runtime error (message in qmv_last_error) */

typedef enum { QMV_MXFP4 = 0, QMV_CB2 = 1, QMV_CB3 = 2, QMV_CB4 = 3, QMV_MXFP8 = 4 } qmv_fmt;

/*
 * Launch flags of qmv_dense_ex, qmv_moe_gather_ex, qmv_moe_gate_up_swiglu and
 * qmv_moe_layer.
 *
 * QMV_FLAG_PREFETCH_INPUTS: the caller guarantees that the weights and the
 * router ids were not written by the kernel immediately preceding this call
 * in the stream (they were ready before it started). The kernel then reads the
 * ids and starts streaming weight tiles while that kernel drains, and waits
 * for it (programmatic dependent launch) only before reading the activations
 * and writing outputs. Typical use: the up and down projections of a MoE
 * layer, whose ids the router produced before the gate projection ran.
 */
#define QMV_FLAG_PREFETCH_INPUTS 1u

/*
 * QMV_FLAG_X_F32 (codebook formats): x_dev holds fp32 activations [nvec][K]
 * (nvec as for the q8_1 buffer it replaces) instead of q8_1. Every CTA
 * quantizes them to q8_1 while staging them in shared memory, with exactly
 * the arithmetic of qmv_quantize_act_q8, so the outputs equal those of
 * qmv_quantize_act_q8 followed by the call, one launch fewer ("DS4 H200:
 * rocmfp2_mix MoE matvec 3.31x ...", "Caveats": the separate q8_1 quantize
 * launch per matvec). Not valid for MXFP4 or qmv_debug_block_sums.
 */
#define QMV_FLAG_X_F32 2u

/*
 * QMV_FLAG_X_F16 (MX formats): activations are fp16 instead of bf16 and every
 * output the call stores is fp16 (h and y of a layer, the combined output of
 * qmv_moe_layer_combine). The products and sums are as for bf16 (exact
 * products, fp32 sums). The f16 MXFP4 gather is the variant mlxcel #2178
 * ("Scope") leaves out of the bf16 arm.
 */
#define QMV_FLAG_X_F16 4u

/*
 * QMV_FLAG_PATH_TENSOR / QMV_FLAG_PATH_CUDA_CORES: override the library's
 * choice between the tcgen05 tensor-core path (dense calls of 5..16 tokens,
 * gathers of 33..QMV_MAX_SLOTS routed slots) and the CUDA-core matvec (one
 * launch, or one per token range of at most QMV_MAX_LAYER_SLOTS slots).
 * Without them the choice follows a cost model measured on GB300: MX dense
 * verify batches and MX gathers of >= 4 slots per distinct expert take the
 * tensor cores; codebook dense batches do when their CUDA-core weight
 * streams (one per 4 tokens) exceed 64 MB, CB4 gathers at >= 8 slots per
 * expert, CB2 / CB3 gathers at >= 12. PATH_TENSOR applies to calls that have a tensor-core form
 * (5..16 dense tokens or 33..128 slots, not fp16 activations, not the
 * gate/up fusion) and is ignored by the others. Not both. Results differ
 * between the two paths only in the order of fp32 additions (integer block
 * sums are identical). For testing and tuning.
 */
#define QMV_FLAG_PATH_TENSOR 8u
#define QMV_FLAG_PATH_CUDA_CORES 16u

/* Limits checked by every entry point. */
#define QMV_MAX_NTOK 16     /* decode / verify tokens per call */
#define QMV_MAX_TOPK 8      /* experts per token */
#define QMV_MAX_SLOTS 128   /* routed (token, slot) pairs of a gather: ntok * top_k */
#define QMV_MAX_LAYER_SLOTS 32  /* routed slots per launch of the CUDA-core gather and gate/up fusion */
#define QMV_MAX_N (1 << 20)
#define QMV_MAX_K (1 << 16)

/*
 * Weight descriptor. `lut` holds the codebook value of code c in lut[c] for
 * the CB formats (entries at or beyond 2^bits are ignored; unused for
 * MXFP4). n_experts = 1 describes a dense matrix.
 */
typedef struct {
  int32_t fmt;        /* qmv_fmt */
  int32_t N;          /* output rows of each matrix, 1 <= N <= QMV_MAX_N */
  int32_t K;          /* reduction length, multiple of 32, <= QMV_MAX_K */
  int32_t n_experts;  /* >= 1 */
  int8_t lut[16];
} qmv_wdesc;

/* Weights per E8M0 scale along K: 32 for MXFP4, MXFP8 and CB4, 16 for CB2 and CB3. */
int32_t qmv_scale_group(int32_t fmt);

/* Bits per weight code: 4, 2, 3, 4, 8 for MXFP4, CB2, CB3, CB4, MXFP8. */
int32_t qmv_code_bits(int32_t fmt);

/*
 * Canonical (storage-order) sizes of ONE expert matrix, in bytes:
 *   codes:  N * K * bits / 8, row-major, each row packed as
 *           MXFP8: element k in byte k;
 *           MXFP4/CB4: element k in byte k/2, low nibble first (a
 *             little-endian uint32 at byte k/2 holds elements k..k+7; mlxcel
 *             #2178, "Proposed Solution" item 1);
 *           CB2: code j of each byte at bits [2j, 2j+2);
 *           CB3: 8 codes per 3 bytes, code j at bits [3j, 3j+3) of the
 *             little-endian 24-bit word (a 16-weight half-block is one
 *             48-bit window; lucebox-hub #21, "Changes" item 2).
 *   scales: N * (K / group) E8M0 bytes, row-major.
 * Return 0 for an invalid descriptor.
 */
size_t qmv_canonical_code_bytes(const qmv_wdesc* desc);
size_t qmv_canonical_scale_bytes(const qmv_wdesc* desc);

/*
 * Size in bytes of the GPU weight layout of one expert (a multiple of 256)
 * and of all n_experts (expert e starts at e * qmv_packed_expert_bytes()).
 * Rows are padded to whole row tiles, so no kernel load goes past the
 * buffer. Return 0 for an invalid descriptor.
 */
size_t qmv_packed_expert_bytes(const qmv_wdesc* desc);
size_t qmv_packed_bytes(const qmv_wdesc* desc);

/*
 * Host packer (offline, not on the timed path). Converts canonical codes
 * [n_experts][canonical code bytes] and E8M0 scales [n_experts][N][K/group]
 * into the GPU weight layout in `out_host` (out_bytes >= qmv_packed_bytes).
 * Padding bytes are zero. The layout is private to this library: upload it
 * unchanged and pass it to qmv_dense / qmv_moe_gather.
 * Errors: QMV_EINVAL (null pointer, bad descriptor), QMV_ESHAPE, QMV_ESIZE.
 */
int qmv_pack_weights(const qmv_wdesc* desc, const uint8_t* codes_host, const uint8_t* scales_host,
                     void* out_host, size_t out_bytes);

/*
 * Inverse of qmv_pack_weights: GPU layout -> canonical codes and scales
 * (same shapes as qmv_pack_weights' inputs). Used to check the packer.
 */
int qmv_unpack_weights(const qmv_wdesc* desc, const void* packed_host, size_t packed_bytes,
                       uint8_t* codes_host, uint8_t* scales_host);

/*
 * q8_1 activation buffer: per vector, K int8 codes followed by K/32 fp16
 * scales d, the vector padded to a multiple of 16 bytes. Vector v starts at
 * v * qmv_act_q8_vec_bytes(K). qmv_act_q8_bytes(nvec, K) is the total.
 */
size_t qmv_act_q8_vec_bytes(int32_t K);
size_t qmv_act_q8_bytes(int32_t nvec, int32_t K);

/*
 * Quantize fp32 activations x_dev [nvec][K] to q8_1 (xq_dev, layout above).
 * Per block of 32, in fp32: amax = max|x|, d = amax / 127, q = x * (1/d)
 * rounded half away from zero and clamped to [-127, 127] (q = 0 when d = 0);
 * d is stored as fp16 (round to nearest even). One launch quantizes every
 * vector (geo-lucebox #31, "Caveats": quantize_q8_1).
 * Errors: QMV_EINVAL, QMV_ESHAPE (K % 32), QMV_EALIGN, QMV_ESIZE, QMV_ECUDA.
 */
int qmv_quantize_act_q8(const float* x_dev, int32_t nvec, int32_t K, void* xq_dev, size_t xq_bytes,
                        void* stream);

/*
 * Host helper: split a q8_1 buffer (host copy) into q [nvec][K] int8 and
 * d [nvec][K/32] fp16 bit patterns.
 */
int qmv_act_q8_unpack(const void* xq_host, int32_t nvec, int32_t K, int8_t* q_host, uint16_t* d_host);

/*
 * Dense decode matvec: y[t] = W . x[t] for t < ntok (1..16; more than a
 * few tokens is a speculative-decoding verify batch, which the pages run
 * through a batched matmul: "perf(ggml/hip): optimize ROCMFPX fp3/fp2 MMVQ on
 * RDNA ...", "Depends on": the batched ROCmFPX MMQ).
 *   w_dev: GPU layout of one matrix (desc->n_experts must be 1).
 *   x_dev: MX formats (MXFP4, MXFP8): bf16 [ntok][K] (fp16 with
 *          QMV_FLAG_X_F16); CB formats: q8_1 buffer of ntok vectors.
 *   y_dev: MX formats: bf16 [ntok][N] (fp16 with QMV_FLAG_X_F16); CB
 *          formats: fp32 [ntok][N].
 * Up to 4 tokens the CUDA-core kernel streams every packed weight byte once
 * per call and applies it to all of them. 5..16 tokens run on the tensor
 * cores (every format; bf16, q8_1 or fp32 activations): the matrix is
 * streamed once, its unscaled elements and the activations are multiplied as
 * f16 with one fp32 accumulator per E8M0 group (exact integer block sums for
 * the codebooks), and the scales are applied in fp32, so every scale byte
 * 0..254 is exact. With fp16 activations (QMV_FLAG_X_F16) 5..16 tokens stream
 * the matrix once per group of 4 tokens, side by side (the DRAM traffic stays
 * about one matrix).
 * Errors: QMV_EINVAL, QMV_ESHAPE, QMV_EALIGN, QMV_ECUDA.
 */
int qmv_dense(const qmv_wdesc* desc, const void* w_dev, const void* x_dev, int32_t ntok, void* y_dev,
              void* stream);

/*
 * MoE expert-gathered decode matvec (the unsorted decode gather):
 *   y[t][j] = W[ids[t][j]] . x(t, j)   for t < ntok, j < top_k,
 * with x(t, j) = x[t] when per_slot_x == 0 (gate/up projections share the
 * token's activation) and x[t * top_k + j] when per_slot_x != 0 (down
 * projection: one activation per slot).
 *   w_dev:   n_experts matrices in GPU layout, expert e at e * qmv_packed_expert_bytes().
 *   ids_dev: int32 [ntok][top_k] expert ids, read on the device. An id outside
 *            [0, n_experts) writes a zero row block (mlxcel #2178,
 *            "Implementation Notes", edge cases). A matrix used by several
 *            (token, slot) pairs is streamed once per call for up to 4 of them.
 *   Up to QMV_MAX_LAYER_SLOTS (32) routed slots the call is the decode
 *   gather above. 33..QMV_MAX_SLOTS (128) slots -- a verify or prefill batch
 *   through a MoE projection -- run as the sorted gather ("perf(ggml/hip):
 *   optimize ROCMFPX fp3/fp2 MMVQ on RDNA ...", "Depends on": the batched MMQ
 *   path) when the slots share experts (ntok * top_k >= 3 * min(n_experts,
 *   ntok * top_k)) and the activations are bf16 (MX) or q8_1 / fp32
 *   (codebooks): the slots are grouped by expert (experts in order of their
 *   first slot, slots in slot order) and each expert's weights are streamed
 *   once per 16 of its slots through the tensor cores, as for qmv_dense. Same
 *   results up to the order of fp32 additions; identical integer block sums.
 *   Otherwise (about one or two slots per expert, or fp16 activations) the
 *   call runs as the decode gather on consecutive token ranges of at most
 *   QMV_MAX_LAYER_SLOTS slots, one launch each (the same bits as those calls
 *   made one by one; an expert used in two ranges is streamed by each).
 *   x_dev:   MX formats: bf16 vectors of K (fp16 with QMV_FLAG_X_F16); CB
 *            formats: q8_1 buffer.
 *   y_dev:   MX formats: bf16 [ntok][top_k][N] (fp16 with QMV_FLAG_X_F16); CB
 *            formats: fp32 [ntok][top_k][N].
 * Errors: QMV_EINVAL (ntok not in 1..16, top_k not in 1..8, ntok * top_k >
 * QMV_MAX_SLOTS), QMV_ESHAPE, QMV_EALIGN, QMV_ECUDA.
 */
int qmv_moe_gather(const qmv_wdesc* desc, const void* w_dev, const void* x_dev, int32_t per_slot_x,
                   const int32_t* ids_dev, int32_t ntok, int32_t top_k, void* y_dev, void* stream);

/* qmv_dense with launch flags (QMV_FLAG_*); flags = 0 is qmv_dense. */
int qmv_dense_ex(const qmv_wdesc* desc, const void* w_dev, const void* x_dev, int32_t ntok, void* y_dev,
                 uint32_t flags, void* stream);

/* qmv_moe_gather with launch flags (QMV_FLAG_*); flags = 0 is qmv_moe_gather. */
int qmv_moe_gather_ex(const qmv_wdesc* desc, const void* w_dev, const void* x_dev, int32_t per_slot_x,
                      const int32_t* ids_dev, int32_t ntok, int32_t top_k, void* y_dev, uint32_t flags,
                      void* stream);

/*
 * Gate and up projections fused with the SwiGLU between them (one launch).
 *
 * Weights: the gate and up matrices of every expert (each N x K, same format,
 * same codebook) packed together by qmv_pack_gate_up into one matrix of
 * 2 * round_up(N, 4) rows per expert, at a stride of
 * qmv_packed_gate_up_expert_bytes(desc). `desc` describes ONE projection
 * (N rows, K columns, n_experts, format, codebook); the packer's inputs are
 * the canonical codes and scales of the gate and up sets in the layout of
 * qmv_pack_weights.
 *
 * qmv_moe_gate_up_swiglu computes, for t < ntok, j < top_k,
 *   g = W_gate[ids[t][j]] . x[t],  u = W_up[ids[t][j]] . x[t],
 *   h[t][j] = silu(g) * u,  silu(z) = z / (1 + exp(-z)),
 * with g and u accumulated in fp32 and never rounded to bf16 (the gpt-oss
 * MoE layer's gate, up and SwiGLU: "perf(rocm): add an mxfp4 arm to the
 * warp-shared gather_qmv kernel for gpt-oss decode", "Problem / Background"
 * and "Current Behavior"). x and h follow qmv_moe_gather with per_slot_x = 0:
 * MX formats: x bf16 [ntok][K], h bf16 [ntok][top_k][N] (both fp16 with
 * QMV_FLAG_X_F16); CB formats: x q8_1, h fp32.
 * An invalid id gives a zero row of h. flags: QMV_FLAG_* (see below). More
 * than QMV_MAX_LAYER_SLOTS routed slots run as one launch per token range of
 * at most that many slots.
 * Errors: as qmv_moe_gather.
 */
size_t qmv_packed_gate_up_expert_bytes(const qmv_wdesc* desc);
int qmv_pack_gate_up(const qmv_wdesc* desc, const uint8_t* gate_codes_host, const uint8_t* gate_scales_host,
                     const uint8_t* up_codes_host, const uint8_t* up_scales_host, void* out_host,
                     size_t out_bytes);
int qmv_moe_gate_up_swiglu(const qmv_wdesc* desc, const void* w_gate_up_dev, const void* x_dev,
                           const int32_t* ids_dev, int32_t ntok, int32_t top_k, void* h_dev, uint32_t flags,
                           void* stream);

/*
 * One MoE decode layer's expert FFN: fused gate/up/SwiGLU, then the down
 * gather on the per-slot h (the gpt-oss layer of "perf(rocm): add an mxfp4
 * arm to the warp-shared gather_qmv kernel for gpt-oss decode", "Problem /
 * Background"; for the codebook formats the DS4 gate/up then down of
 * "DS4 H200: rocmfp2_mix MoE matvec 3.31x + ROCmFP4 dense matvec 1.53x",
 * "Caveats", with h quantized to q8_1 in between).
 *   y[t][j] = W_down[ids[t][j]] . h[t][j],  h as qmv_moe_gate_up_swiglu.
 * gate_up_desc: one projection (N, K); down_desc: (N_down, K = N). Both MX
 * formats (MXFP4 and MXFP8 may be mixed) or both codebook formats, same
 * n_experts. x as qmv_moe_gate_up_swiglu.
 * y: MX formats bf16 [ntok][top_k][N_down] (fp16 with QMV_FLAG_X_F16);
 * codebooks fp32.
 * Two launches (more for more than QMV_MAX_LAYER_SLOTS routed slots, up to
 * QMV_MAX_SLOTS, as qmv_moe_gather and qmv_moe_gate_up_swiglu split them):
 * the fused gate/up/SwiGLU gather stores h in the workspace (MX formats bf16
 * or fp16, codebooks fp32), then the down gather reads the per-slot h
 * (codebooks: it quantizes h to q8_1 while staging it, as QMV_FLAG_X_F32).
 * workspace: caller-owned device scratch of at least
 * qmv_moe_layer_workspace_bytes(gate_up_desc, ntok, top_k) bytes, 16-byte
 * aligned; its contents on entry do not matter. Calls that share a workspace
 * must be ordered on one stream.
 * flags apply to the gate/up launch (QMV_FLAG_X_F32: a codebook layer's x is
 * fp32; QMV_FLAG_X_F16: an MX layer's x, h and y are fp16); the down gather
 * always prefetches its weights and ids (they were complete before the
 * layer's first launch).
 */
size_t qmv_moe_layer_workspace_bytes(const qmv_wdesc* gate_up_desc, int32_t ntok, int32_t top_k);
int qmv_moe_layer(const qmv_wdesc* gate_up_desc, const void* w_gate_up_dev, const qmv_wdesc* down_desc,
                  const void* w_down_dev, const void* x_dev, const int32_t* ids_dev, int32_t ntok, int32_t top_k,
                  void* workspace_dev, size_t workspace_bytes, void* y_dev, uint32_t flags, void* stream);

/*
 * Router-weighted combine of a MoE layer's per-slot outputs:
 *   y[t][n] = sum over j with ids[t][j] in [0, E) of weights[t][j] * ys[t][j][n]
 * (fp32 fma in slot order, the same order every run). The pages print the
 * switch-GLU part of the gpt-oss layer (per-slot outputs of the top-k experts,
 * "perf(rocm): add an mxfp4 arm to the warp-shared gather_qmv kernel for
 * gpt-oss decode", "Current Behavior": GptOssSwitchGLU); weighting and summing
 * them is the MoE block's combine (a reading: the pages do not print it).
 * down_desc: the down projection (N outputs, n_experts, format: MX formats
 * -> ys and y bf16, codebooks -> fp32). ys [ntok][top_k][N] (as qmv_moe_layer's
 * y), weights fp32 [ntok][top_k], ids int32 [ntok][top_k], y [ntok][N]; all
 * on the device, 16-byte aligned. One launch (dependent launch after the
 * kernel that wrote ys).
 * Errors: QMV_EINVAL, QMV_ESHAPE, QMV_EALIGN, QMV_ECUDA.
 */
int qmv_moe_combine(const qmv_wdesc* down_desc, const void* ys_dev, const float* weights_dev,
                    const int32_t* ids_dev, int32_t ntok, int32_t top_k, void* y_dev, void* stream);

/* qmv_moe_combine with flags: QMV_FLAG_X_F16 (MX formats) makes ys and y
 * fp16; flags = 0 is qmv_moe_combine. */
int qmv_moe_combine_ex(const qmv_wdesc* down_desc, const void* ys_dev, const float* weights_dev,
                       const int32_t* ids_dev, int32_t ntok, int32_t top_k, void* y_dev, uint32_t flags,
                       void* stream);

/*
 * qmv_moe_layer followed by qmv_moe_combine: the layer's combined output
 * y [ntok][N_down] (MX formats bf16, or fp16 with QMV_FLAG_X_F16; codebooks
 * fp32) for router weights
 * weights_dev fp32 [ntok][top_k]. The per-slot outputs live in the workspace,
 * which needs qmv_moe_layer_combine_workspace_bytes(...) bytes (the layer's
 * workspace followed by ntok * top_k * N_down outputs). Three launches.
 */
size_t qmv_moe_layer_combine_workspace_bytes(const qmv_wdesc* gate_up_desc, const qmv_wdesc* down_desc,
                                             int32_t ntok, int32_t top_k);
int qmv_moe_layer_combine(const qmv_wdesc* gate_up_desc, const void* w_gate_up_dev, const qmv_wdesc* down_desc,
                          const void* w_down_dev, const void* x_dev, const int32_t* ids_dev,
                          const float* weights_dev, int32_t ntok, int32_t top_k, void* workspace_dev,
                          size_t workspace_bytes, void* y_dev, uint32_t flags, void* stream);

/*
 * qmv_moe_layer for callers that cannot allocate device memory. (No
 * counterpart on the pages this library follows; it exists for how the
 * library is embedded.) Some callers may not allocate GPU memory while they
 * decode: an inference server that gives the whole device to its own memory
 * pool before serving, a plugin living in another application's CUDA context
 * under a fixed budget, or code running while a stream is being captured,
 * where allocating is not allowed. This entry point takes the same arguments
 * as qmv_moe_layer minus the workspace and uses a static scratch array of
 * QMV_NOALLOC_SCRATCH_BYTES bytes compiled into the library instead; it calls
 * no allocator.
 *  - Every GPU that loads the library holds the array until the process exits.
 *  - The array's device address belongs to a CUDA context. The first call in
 *    each context (the device's primary context, a context the host
 *    application made itself, or the primary context created again after
 *    cudaDeviceReset) looks it up, with that context current, and keeps it
 *    for later calls in the same context; make that first call before any
 *    stream capture.
 *  - A layer whose qmv_moe_layer_workspace_bytes exceeds the array is rejected
 *    with QMV_ESIZE (use qmv_moe_layer with a workspace for it).
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it needs to start at zero: every byte the layer reads from it
 *    is written earlier in the same call. Calls that can overlap on the GPU
 *    (other streams, other host threads) race on the array: order them.
 */
#define QMV_NOALLOC_SCRATCH_BYTES (1u << 20)
int qmv_moe_layer_noalloc(const qmv_wdesc* gate_up_desc, const void* w_gate_up_dev, const qmv_wdesc* down_desc,
                          const void* w_down_dev, const void* x_dev, const int32_t* ids_dev, int32_t ntok,
                          int32_t top_k, void* y_dev, uint32_t flags, void* stream);

/*
 * SwiGLU between the gate/up and down gathers of a gpt-oss-style MoE layer:
 * h[i] = silu(g[i]) * u[i], silu(z) = z / (1 + exp(-z)), bf16 in and out,
 * fp32 arithmetic, n elements ("perf(rocm): add an mxfp4 arm ...", "Problem /
 * Background": 24 layers times gate, up and down).
 * Errors: QMV_EINVAL, QMV_EALIGN, QMV_ECUDA.
 */
int qmv_swiglu_bf16(const void* g_dev, const void* u_dev, void* h_dev, int64_t n, void* stream);

/*
 * Test export: the same kernels as qmv_dense / qmv_moe_gather for the CB
 * formats, additionally writing every integer block sum
 *   sums[slot][n][h] = sum_{i in h} lut[c_{n,i}] * q_i      (int32)
 * with h a 16-weight half-block (CB2, CB3) or 32-weight block (CB4), slot =
 * t (dense) or t * top_k + j (gather), sums_bytes >= slots * N * (K/span) * 4.
 * ids_dev = NULL selects the dense path (top_k and per_slot_x ignored).
 * Slots with an invalid id are left untouched.
 */
int qmv_debug_block_sums(const qmv_wdesc* desc, const void* w_dev, const void* x_dev,
                         int32_t per_slot_x, const int32_t* ids_dev, int32_t ntok, int32_t top_k,
                         void* y_dev, int32_t* sums_dev, size_t sums_bytes, void* stream);
/* qmv_debug_block_sums with launch flags (QMV_FLAG_PREFETCH_INPUTS,
 * QMV_FLAG_PATH_*). */
int qmv_debug_block_sums_ex(const qmv_wdesc* desc, const void* w_dev, const void* x_dev,
                            int32_t per_slot_x, const int32_t* ids_dev, int32_t ntok, int32_t top_k,
                            void* y_dev, int32_t* sums_dev, size_t sums_bytes, uint32_t flags, void* stream);

/*
 * Test export (host only, no device needed): the CUDA-core matvec's launch
 * plan for a call shape and an explicit device shape (sm_count SMs,
 * ctas_per_sm CTAs per SM, smem_per_sm bytes of shared memory per SM). out
 * (>= 12 entries): vectors per entry, warps per CTA, ring stages, item upper
 * bound, grid, K splits, chunks per split, items per CTA, activation vectors
 * staged per CTA, contiguous dealing (0/1), dynamic shared memory bytes, row
 * tiles. gather != 0 describes an expert gather (per_slot_x as there).
 * Errors: QMV_EINVAL, QMV_ESHAPE, QMV_ESIZE.
 */
int qmv_debug_plan(const qmv_wdesc* desc, int32_t ntok, int32_t top_k, int32_t gather, int32_t per_slot_x,
                   uint32_t flags, int32_t sm_count, int32_t ctas_per_sm, int64_t smem_per_sm, int64_t* out,
                   int32_t n_out);

/*
 * Test export (host only, no device needed): the path a call of this shape
 * and these flags takes (QMV_FLAG_PATH_* included). out (>= 2 entries):
 * out[0] = 1 for the tcgen05 tensor-core kernels (verify batch or sorted
 * gather), 0 for the CUDA-core matvec; out[1] = tokens per CUDA-core launch
 * (ntok, or QMV_MAX_LAYER_SLOTS / top_k for a gather of more routed slots).
 * gather != 0 describes an expert gather; glu != 0 the fused gate/up
 * (qmv_moe_gate_up_swiglu). Errors: QMV_EINVAL, QMV_ESIZE.
 */
int qmv_debug_path(const qmv_wdesc* desc, int32_t ntok, int32_t top_k, int32_t gather, int32_t glu,
                   uint32_t flags, int64_t* out, int32_t n_out);

/*
 * Test export: decode the GPU weight layout of one matrix with the kernels'
 * device decode routines to fp32 w_dev [N][K] = value(code) * 2^(e-127).
 * For the CB formats value(code) = lut[code].
 */
int qmv_debug_dequant(const qmv_wdesc* desc, const void* w_dev, int32_t expert, float* out_dev,
                      size_t out_bytes, void* stream);

/*
 * Device-side status: bit flags set by kernels whose bounded waits gave up:
 * 1 (not used), 2 weight tile copy, 4 copy still in flight when giving
 * up, 8 the wait probe; and 16: a CTA of a per-slot gather needed more
 * staged activation vectors than the launch planned for (a library bug; the
 * outputs of that call are wrong). No kernel here waits on another kernel, so
 * bits 1-4 indicate a lost asynchronous copy. Synchronizes the device;
 * clear != 0 resets the flags.
 */
int qmv_device_status(uint32_t* flags_host, int32_t clear);

/*
 * Test export: launches one CTA that waits, with the kernels' bounded wait and
 * the given limit (0 < limit_ns <= 1 s), on an mbarrier phase that nothing
 * completes. The wait gives up, the kernel sets status bit 8 and returns; the
 * context stays usable. Checks the timeout path without a fault or a hang.
 */
int qmv_debug_wait_probe(uint64_t limit_ns, void* stream);

/*
 * Diagnostic export: the compute rate of the matvec's inner loop. Launches
 * (SM count x ctas_per_sm) CTAs of the production launch shape for nv
 * activation vectors (1..4) in which every warp applies the format's chunk
 * routine (decode, products, block sums and scales of 8 rows x 1024 columns)
 * `iters` times to a tile held in shared memory, with no copies or waits, so
 * that its weights per clock per SM can be compared with the rate the weight
 * stream delivers (the secondary ALU roofline). *weights_host = matrix
 * weights one launch processes (each applied to nv vectors), *threads_host =
 * threads launched; sink_dev (fp32 [threads], 16-byte aligned) receives one
 * value per thread so that nothing is optimized away. sink_dev = NULL only
 * reports the two counts. Time the launch with events on `stream`.
 * Errors: QMV_EINVAL, QMV_EALIGN, QMV_ESIZE, QMV_ECUDA.
 */
int qmv_debug_chunk_rate(int32_t fmt, int32_t nv, int32_t ctas_per_sm, int32_t iters, float* sink_dev,
                         size_t sink_bytes, int64_t* weights_host, int64_t* threads_host, void* stream);

/*
 * Diagnostic exports of the phase probe, a build variant of this library
 * (bit_quantized_moe_gb300/build.py --phase-probe defines QMV_PHASE_PROBE):
 * lane 0 of every warp of the CUDA-core matvec records %globaltimer (ns) at
 * fixed phases of its launch -- kernel start, work list built, tile copies
 * issued before griddepcontrol.wait, the wait returned, activation loads
 * issued, every ring stage's first copy issued, activations staged, first
 * tile landed and computed, second and third tiles landed, last tile
 * computed, warp done -- into a per-format buffer of
 * qmv_debug_phase_entries() uint64 values laid out [launch slot 0..7][CTA
 * 0..511][warp 0..15][phase 0..15], 0 where nothing was recorded.
 * qmv_debug_phase_probe(1) makes the following launches record (slots dealt
 * in launch order, modulo 8; a CUDA graph keeps the slots of its capture);
 * qmv_debug_phase_read copies one format's buffer to the host (synchronizes)
 * and clears it if `clear`. In the product build both return QMV_EINVAL.
 */
size_t qmv_debug_phase_entries(void);
int qmv_debug_phase_probe(int32_t enable);
int qmv_debug_phase_read(int32_t fmt, uint64_t* out_host, size_t n, int32_t clear);

/* Message of the last failure on the calling thread ("" if none). */
const char* qmv_last_error(void);

/* Library version string. */
const char* qmv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QMV_H */
