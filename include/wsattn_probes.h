/*
 * wsattn_probes.h -- C ABI of libwsattn_probes.so, the test-only library of
 * single-tile kernels that check the building blocks of the attention kernel
 * in isolation: the first tensor-core stage S = Q K^T and the second stage
 * O = P V of the attention loop in "Tawa: Automatic Warp Specialization for
 * Modern GPUs with Asynchronous References", Section III-D, Algorithm 1, each
 * run once on one 128-row tile with the same TMA boxes, shared-memory
 * descriptors and instruction descriptors as the attention kernel.
 *
 * All pointers are device pointers, 16-byte aligned; the calls synchronise the
 * device.  Return: 0 ok, 1 bad pointer, 2 unsupported D (only 64 and 128),
 * 3 CUDA error, 4 a device-side wait gave up (bounded waits, no hang).
 */
#ifndef WSATTN_PROBES_H_
#define WSATTN_PROBES_H_

#ifdef __cplusplus
extern "C" {
#endif

/* c[128][128] (fp32, row-major) = a[128][D] * b[128][D]^T; a, b 16-bit row-major
 * (f16, or bf16 when bf16 != 0). */
int wsa_probe_qk(const void* a, const void* b, float* c, int D, int bf16);

/* o[128][D] (fp32, row-major) = p[128][128] * v[128][D]; p and v 16-bit row-major.
 * p is written to Tensor Memory with tcgen05.st (two values per column) and fed
 * to the TMEM-operand form of tcgen05.mma; v is read as an MN-major operand. */
int wsa_probe_pv(const void* p, const void* v, float* o, int D, int bf16);

/* The 8-bit forms (tcgen05.mma.kind::f8f6f4, E4M3 operands, K = 32 per
 * instruction) on one 128 x 128 x 128 tile:
 *   c[128][128] = a[128][128] * b[128][128]^T           (both K-major, SMEM)
 *   o[128][128] = p[128][128] * vt[128][128]^T           (p from TMEM, four
 *                                                          values per column)
 * a, b, p, vt: E4M3 bytes, row-major; vt is V transposed (vt[d][key]). */
int wsa_probe_qk_e4m3(const void* a, const void* b, float* c);
int wsa_probe_pv_e4m3(const void* p, const void* vt, float* o);

/* The two shared-memory forms of the backward pass, one 128 x 128 x D tile
 * (16-bit, D = 64 or 128; bf16 when bf16 != 0), c fp32 row-major [128][D]:
 *   wsa_probe_kmaj_mn: c = a b,  a[128][128] row-major (read K-major),
 *                                b[128][D] row-major (read MN-major)
 *   wsa_probe_mn_mn:   c = at^T b, at[128][128] row-major holding A
 *                                transposed (read MN-major), b as above */
int wsa_probe_kmaj_mn(const void* a, const void* b, float* c, int D, int bf16);
int wsa_probe_mn_mn(const void* at, const void* b, float* c, int D, int bf16);

#ifdef __cplusplus
}
#endif

#endif /* WSATTN_PROBES_H_ */
