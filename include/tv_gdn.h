/*
 * tv_gdn.h -- rollback-free tree verification of a Gated DeltaNet (GDN) layer
 * and the deferred commit of its recurrent state.
 *
 * Source: "Technische Samenvatting: Trees from Marginals (DFlash-TfM)",
 * "3. Rollback-vrije Boom-verificatie voor GDN".  A GDN layer updates its
 * state by
 *     S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
 * S a d_k x d_v matrix.  Verifying a draft tree gives every node the output
 * o_t = S_t^T q_t of the state reached along its own root-to-node path, in one
 * pass and without touching the committed state S_0; the state is committed
 * once the accepted branch is known.  With u_t = beta_t (v_t - alpha_t
 * S_parent^T k_t) and g_t the product of alpha along the path,
 *     S_t = g_t S_0 + sum over ancestors-or-self i of (g_t / g_i) k_i u_i^T,
 * so the pseudo-values U solve the triangular system (I + X) U = beta *
 * (V - g * K S_0) with X_ti = beta_t (g_t / g_i) k_t . k_i on the node's strict
 * ancestors (the page's "(I+X)U = beta V", its X the ancestor-masked
 * interaction matrix), and O = g * (Q S_0) + Y U with Y_ti = (g_t / g_i)
 * q_t . k_i on ancestors-or-self.
 *
 * Layouts (row-major):
 *   state   float32 [B, Hv, dv, dk]   S^T: row j holds column j of S
 *   q, k    bf16    [B, N, Hk, dk]    value head h reads key head h / (Hv / Hk)
 *   v       bf16    [B, N, Hv, dv]
 *   alpha   float32 [B, N, Hv]        decay, in (0, 1]
 *   beta    float32 [B, N, Hv]        write strength
 *   anc     uint64  [B, N]            ancestor-or-self bitmask (tv_build_ancestors)
 * d_k is a multiple of 32 and d_v of 64, both at most 128; N <= 64; Hv % Hk == 0.
 * Conventions are those of tv.h.
 */
#ifndef TV_GDN_H_
#define TV_GDN_H_

#include "tv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * tv_gdn_tree_verify -- outputs of every tree node from the committed state.
 *   out     float32 [B, N, Hv, dv]   o_t = S_t^T q_t
 *   u       float32 [B, N, Hv, dv]   pseudo-values, kept for tv_gdn_commit
 *   g       float32 [B, N, Hv]       product of alpha along each node's path
 *   kernel  0 auto, 1 CUDA cores (fp32 FMA), 2 tensor cores (tcgen05; d_k 64
 *           or 128; one CTA per sequence, value head and 64 columns of d_v),
 *           3 tensor cores, persistent pipeline (one CTA per SM over the
 *           (sequence, value head) problems, the next state in flight while
 *           the current one is solved; d_k 64 or 128 and N <= 32).  Auto takes
 *           3, else 2, else 1.  On the tensor cores K and Q enter as the bf16
 *           they are and the fp32 state as three bf16 planes (hi + mid + lo,
 *           24 significant bits), with fp32 accumulation: every kernel gives
 *           fp32-accurate products.
 *   status  int32   [B]              sequences with a non-zero status (a
 *                                    malformed tree) are skipped: their outputs
 *                                    are left untouched; a wait of the
 *                                    tensor-core kernel that runs past its
 *                                    bound (never on a healthy GPU) writes
 *                                    TV_ERR_CUDA
 * Errors: TV_ERR_ARG (NULL pointers, sizes out of range), TV_ERR_UNSUPPORTED
 * (kernel 2 with d_k not 64 or 128; kernel 3 with d_k not 64 or 128 or N > 32).
 */
tv_status tv_gdn_tree_verify(const float *state, const void *q, const void *k, const void *v,
                             const float *alpha, const float *beta, const uint64_t *anc, int B,
                             int N, int Hk, int Hv, int dk, int dv, float *out, float *u, float *g,
                             int kernel, int32_t *status, tv_stream stream);

/*
 * tv_gdn_commit -- the state after the accepted path acc_nodes[b][0 .. n_acc[b]):
 *     state_out = g_l S_0 + sum over the path of (g_l / g_p) k_p u_p^T,
 * l the last accepted node (tv_tree_walk's acc_nodes / n_acc; u from
 * tv_gdn_tree_verify).  g_l / g_p is formed as the product of alpha over the
 * path nodes after p, so no division is made.  n_acc = 0, a node index out of
 * range or a non-zero status copies S_0.  state_out may not alias state_in.
 * state_in, state_out, k and u must be 16-byte aligned (the state moves in
 * bulk copies of whole 32-row tiles, k and u rows in 16-byte pieces).
 * Errors: TV_ERR_ARG (NULL pointers, sizes out of range, aliasing, alignment).
 */
tv_status tv_gdn_commit(const float *state_in, const void *k, const float *u, const float *alpha,
                        const int32_t *acc_nodes, const int32_t *n_acc, int B, int N, int Hk,
                        int Hv, int dk, int dv, float *state_out, const int32_t *status,
                        tv_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TV_GDN_H_ */
