/*
 * spark_layer.h -- C ABI of the rest of a spark2_5 decoder layer (the MLP
 * half) and of the model's head, for NVIDIA GB300 (sm_103a).  Same library
 * and conventions as spark_attn.h (device pointers owned by the caller,
 * 16-byte aligned; work enqueued on `stream`; SPARK_OK or a negative
 * spark_status).
 *
 * turbospark-runtime 0.3.0, src/families/spark/mod.rs: the module doc's
 * transcription of one decoder layer ends, after the attention block's raw
 * residual add, with
 *
 *   x      = h / sqrt(mean(h^2) + eps) * post_attention_layernorm   (plain w)
 *   h      = h + down_proj @ (gelu_erf(gate_proj @ x) * (up_proj @ x))
 *
 * and the model with
 *
 *   x      = h / sqrt(mean(h^2) + eps) * model.norm
 *   logits = embed_tokens @ x            (the head tied to the embedding)
 *
 * gelu_erf(z) = z * Phi(z) = z / 2 * (1 + erf(z / sqrt 2)), the exact GELU.
 * produce_real_spark's layer loop runs the second norm and then
 * mlp::encode_mlp_block, whose residual add closes the layer; after the last
 * layer the final norm and one GEMV over the embedding rows give the logits.
 * The sizes `intermediate` and `vocab` are the model's (arch.intermediate_size,
 * arch.vocab_size); the pages do not print them, so they are arguments here.
 */
#ifndef SPARK_LAYER_H
#define SPARK_LAYER_H

#include "spark_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The MLP half of one layer (device, caller-owned), all of element type
 * `dtype` (spark_dtype):
 *   norm_w  [hidden]                  post_attention_layernorm.weight
 *   gate_w  [intermediate][hidden]    mlp.gate_proj.weight
 *   up_w    [intermediate][hidden]    mlp.up_proj.weight
 *   down_w  [hidden][intermediate]    mlp.down_proj.weight
 * intermediate: a multiple of 8 in [8, 16384]. */
typedef struct spark_mlp_weights {
  const void* norm_w;
  const void* gate_w;
  const void* up_w;
  const void* down_w;
  int32_t intermediate;
  int32_t dtype;
} spark_mlp_weights;

/* Bytes of device workspace spark_mlp_decode needs for `batch` sequences at
 * this intermediate size (0 for invalid arguments); intermediate == 0 sizes a
 * workspace for spark_head_logits alone.  The workspace holds the GELU
 * products, the tensor-core path's activation rows (hi, lo), its split-K
 * partial results and tickets, and the device error word (its first 4 bytes,
 * read and cleared by spark_attn_error_word).  Initialise it once with
 * spark_attn_workspace_init.  A workspace sized for an intermediate size also
 * serves spark_head_logits; it is not shared with the spark_attn_* calls. */
size_t spark_mlp_workspace_bytes(const spark_geom* g, int32_t intermediate, int32_t batch);

/* The MLP half of one decoder layer for `batch` independent sequences.
 *   h      [batch][hidden] fp32 device: the residual stream after the
 *          attention block.
 *   out    [batch][hidden] fp32 device: h + down_proj(...).  May equal h.
 *   path   SPARK_PATH_* (spark_attn.h): AUTO takes the GEMV kernels for
 *          batch <= 4 or fp32 weights, else the tensor-core GEMMs (bf16
 *          weights, hidden % 64 == 0); GEMV / MMA force one (MMA on fp32
 *          weights is UNSUPPORTED).
 *   workspace >= spark_mlp_workspace_bytes(g, w->intermediate, batch) bytes,
 *          256-byte aligned, initialised once; calls sharing a workspace
 *          must be ordered on one stream.
 * Errors: INVALID_ARG, WORKSPACE, UNSUPPORTED before any work is enqueued;
 * CUDA if a launch fails. */
int spark_mlp_decode(const spark_geom* g, const float* h, const spark_mlp_weights* w,
                     int32_t batch, float* out, int32_t path, void* workspace,
                     size_t workspace_bytes, void* stream);

/* The head: final RMSNorm and the logits of the tied embedding.
 *   h       [batch][hidden] fp32 device: the residual stream after the last
 *           layer.
 *   norm_w  [hidden] model.norm.weight, element type `dtype`.
 *   embed   [vocab][hidden] embed_tokens.weight, element type `dtype`.
 *   vocab   a multiple of 8 in [8, 2^22].
 *   logits  [batch][vocab] fp32 device.
 *   path    as for spark_mlp_decode.
 *   workspace >= spark_mlp_workspace_bytes(g, 0, batch), initialised once.
 * Errors as spark_mlp_decode. */
int spark_head_logits(const spark_geom* g, const float* h, const void* norm_w,
                      const void* embed, int32_t vocab, int32_t dtype, int32_t batch,
                      float* logits, int32_t path, void* workspace, size_t workspace_bytes,
                      void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SPARK_LAYER_H */
