/*
 * mla_workload.h -- device-side generator of the seeded synthetic inputs.
 *
 * Not part of the method: the pages publish no dataset, so the benchmark and the
 * tests draw synthetic latent rows. The long-context pools (61 layers x 184,352
 * rows x 1152 B, about 13 GB; "The Moment of Doubt", subject message: about 13 GB
 * of KV per step at 185k) are too large to draw on the host, so the library can
 * draw them in place with the same counter-based recipe the host generator uses:
 *
 *   h_i = SplitMix64 output for state seed + (i + 1) * 0x9E3779B97F4A7C15 (mod 2^64)
 *   x_i = (sum of the four 16-bit fields of h_i - 131070) * float32(0x37DDB3D7)
 *   dst[i] = x_i rounded to bf16, round-to-nearest-even
 *
 * (an Irwin-Hall approximation of N(0,1); every step is integer work or one
 * correctly rounded float32 multiply, so host and device agree bit for bit).
 */
#ifndef MLA_WORKLOAD_H
#define MLA_WORKLOAD_H

#include <stdint.h>

#include "mla_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mla_fill_normal_bf16 -- dst[i] = draw(seed, start + i) for i in [0, count).
 *   dst    device bf16 array of `count` elements, 2-byte aligned.
 *   seed   stream seed; start: counter of dst[0].
 * Enqueued on `stream`; allocates nothing. Returns MLA_OK, MLA_ERR_INVALID_ARGUMENT
 * (null dst with count > 0, negative count or start) or MLA_ERR_CUDA.
 */
int mla_fill_normal_bf16(void *dst, int64_t count, uint64_t seed, uint64_t start, mla_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_WORKLOAD_H */
