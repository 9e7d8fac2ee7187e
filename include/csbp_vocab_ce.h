/*
 * csbp_vocab_ce.h -- C ABI of libcsbp's streamed LM-head cross-entropy:
 * the vocabulary loss of block-diffusion training and of drafter training,
 * forward and backward in one call, on one sm_103a GPU.
 *
 * Method (Turbo-dLLM project page "Block Parallelism for Efficient
 * Distributed Long-Context Diffusion Language Model Training", section
 * "Library", tables "Speculative Decoding Optimizations" and "Block Diffusion
 * Optimizations", row "Vocabulary loss"): hidden rows go through the LM head
 * in token chunks and the cross-entropy is taken without the logits of the
 * whole sequence ever existing; the drafter's head is frozen.  Per row i
 * with hidden state h_i, head W [V][Dm] and target t_i:
 *
 *   z_i    = W h_i,   lse_i = log sum_v exp(z_iv),   loss_i = lse_i - z_{i,t_i}
 *   g_i    = s (softmax(z_i) - onehot(t_i))
 *   dH_i   = g_i W,   dW = sum_i g_i^T h_i   (dW only for a trained head)
 *
 * s is the caller's gradient scale (dObjective/dloss_i of every counted row,
 * e.g. 1/number of counted rows).  A row with t_i < 0 is ignored: its loss
 * and gradient are 0 and it adds nothing to dW.
 *
 * Conventions are those of csbp.h: caller-owned memory, asynchronous work on
 * `stream`, errors as csbp_status before anything is enqueued, 16-byte
 * aligned device pointers, and a device status word at the start of the
 * workspace (zero it once after allocating; csbp_check_status reads and
 * clears it).
 */
#ifndef CSBP_VOCAB_CE_H_
#define CSBP_VOCAB_CE_H_

#include <stddef.h>
#include <stdint.h>

#include "csbp.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct csbp_ce_problem {
  int64_t rows;        /* N >= 1: rows whose loss is taken                        */
  int32_t d_model;     /* Dm: hidden size; multiple of 64, 64 .. 65536            */
  int32_t vocab;       /* V: vocabulary size; multiple of 64, 64 .. 2^24          */
  int32_t chunk_rows;  /* C: rows per chunk, a multiple of 128 (0: 8192); the
                          logits of at most C rows exist at any time            */
  int32_t head_grad;   /* 1: also write dW (trained head); 0: frozen head         */
  float grad_scale;    /* s (finite)                                              */
} csbp_ce_problem;

/* Workspace bytes csbp_vocab_ce needs for this problem: the status word,
 * fp32 logits [C][V], bf16 g [C][V], per-row partial (max, sum) of each
 * 256-column vocabulary tile and the target logits.  0 if the problem is
 * invalid. */
size_t csbp_ce_workspace_bytes(const csbp_ce_problem* problem);

/* Loss, LSE and gradients of the problem, chunk by chunk on `stream`.
 *  h       device bf16 [N][Dm]            hidden rows
 *  w       device bf16 [V][Dm]            LM head
 *  target  device int32 [N]               class per row; < 0 (or >= V) ignores
 *                                         the row
 *  loss    device fp32 [N]  (out)         lse_i - z_{i,t_i}, 0 when ignored
 *  lse     device fp32 [N]  (out)         natural-log softmax denominator
 *  dh      device bf16 [N][Dm] (out)      gradient of the objective w.r.t. h
 *  dw      device fp32 [V][Dm] (out)      gradient w.r.t. W (overwritten);
 *                                         must be NULL when head_grad == 0
 *  workspace, workspace_bytes             >= csbp_ce_workspace_bytes
 * Returns CSBP_ERR_INVALID for a bad shape, pointer or alignment,
 * CSBP_ERR_WORKSPACE if the workspace is too small, CSBP_ERR_CUDA if a launch
 * fails. */
csbp_status csbp_vocab_ce(const csbp_ce_problem* problem, const void* h, const void* w,
                          const int32_t* target, float* loss, float* lse, void* dh, float* dw,
                          void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CSBP_VOCAB_CE_H_ */
