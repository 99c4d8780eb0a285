/*
 * polar.h — C ABI of the Polar Express orthogonalisation in libswa_attn.so (B300, sm_103a).
 *
 * The Muon optimiser step of the habr "Autoresearch" deep dive (train.py listing, optimiser section,
 * muon_step_fused with polar_express_coeffs) orthogonalises each momentum-mixed gradient matrix G:
 *   X = G / (||G||_F * 1.02 + 1e-6)
 *   for each of the first `steps` coefficient triples (a, b, c) of the listing's table:
 *     wide (rows <= cols): A = X X^T, B = b A + c A A, X = a X + B X
 *     tall (rows > cols):  A = X^T X, B = b A + c A A, X = a X + X B
 * which maps every singular value s of X to a s + b s^3 + c s^5 (so X tends to U V^T). The listing
 * runs it on bf16 tensors; here every product takes bf16 operands, accumulates in fp32 on the tensor
 * cores and rounds its result to bf16 once, together with its linear term:
 *   A = bf16(X X^T),  B = bf16(c (A A) + b A),  X' = bf16(a X + B X)      (tall: X^T X and X B)
 * and the normalisation rounds as the listing's bf16 operations do: nrm = bf16(||G||_F) (fp32 sum),
 * den = bf16(bf16(nrm * 1.02) + 1e-6), X = bf16(G / den).
 *
 * Conventions: matrices are device pointers to bf16, a batch of `batch` row-major m x n matrices
 * stored back to back ([batch, m, n]); m and n are multiples of 8 (rows start on 16-byte boundaries),
 * pointers 16-byte aligned. Calls are asynchronous on `stream` and return ATTN_OK or an ATTN_ERR_*
 * code of attn.h (attn_init must have succeeded; a bounded wait that gives up is reported through
 * attn_device_status).
 */
#ifndef SWA_POLAR_H
#define SWA_POLAR_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* pe_workspace_bytes — scratch pe_normalize / pe_step / polar_express need: A and B ([batch, s, s],
 * s = min(m, n)), one more [batch, m, n] matrix and the normalisation's fp32 partial sums (at most
 * 1024 per matrix), each on a 256-byte boundary. 0 for a non-positive size. */
size_t pe_workspace_bytes(int batch, int m, int n);

/* pe_step_flops — the FLOPs one pe_step on this shape executes on the tensor cores (2 K per output
 * element of the tiles its three products compute; A and B only on and above the diagonal), for
 * roofline accounting on the current device. 0 for an invalid shape or before attn_init. The method's
 * own count (the listing's products in full) is 4 s^2 l + 2 s^3 per matrix (s, l = min, max of m, n). */
double pe_step_flops(int batch, int m, int n);

/* pe_normalize — X = G / (||G||_F * 1.02 + 1e-6) per matrix (bf16 steps as above). X may equal G
 * (in place); otherwise G and X must not overlap, and neither may overlap the workspace (at least
 * pe_workspace_bytes(batch, m, n) bytes, 256-byte aligned). The sum of squares is taken in fp32 over
 * chunks whose partial sums are added in one fixed order: the result is deterministic. */
int pe_normalize(const void* G, void* X, int batch, int m, int n, void* workspace, size_t workspace_bytes,
                 void* stream);

/* pe_step — one step with the listing's coefficient triple number `step` (0..4): Y from X. X and Y
 * must not overlap each other or the workspace. A and B are symmetric: only their 128 x 128 blocks on
 * and above the diagonal are computed, and the products that read them take a block below the
 * diagonal as the transpose of its mirror. After the call (when the stream reaches it) the workspace
 * starts with that step's A and then B ([batch, s, s] bf16 each, s = min(m, n)); their blocks below
 * the diagonal hold no data. */
int pe_step(const void* X, void* Y, int batch, int m, int n, int step, void* workspace, size_t workspace_bytes,
            void* stream);

/* polar_express — pe_normalize then steps 0 .. steps-1 (steps 0..5; the listing uses 5), result in X.
 * G is not modified; X must not overlap G or the workspace. */
int polar_express(const void* G, void* X, int batch, int m, int n, int steps, void* workspace,
                  size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SWA_POLAR_H */
