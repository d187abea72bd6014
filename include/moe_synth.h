/*
 * moe_synth.h -- C ABI of libmoe_synth.so: the device twin of the seeded
 * synthetic-input generator (moe_decode_quantized_gb300/synth.py). It fills
 * device memory with exactly the bytes the host generator produces, so the
 * multi-GB expert arenas can be made in place. It is test and benchmark
 * infrastructure, holds none of the layer's arithmetic, and has no
 * counterpart on the reference pages.
 *
 * Generator: SplitMix64 in counter mode; word i of the tensor keyed `key` is
 * mix64(key + (i + 1) * 0x9E3779B97F4A7C15). Keys come from the host module
 * (synth.tensor_key). All calls enqueue on `stream` and return 0 or a CUDA
 * error code (cudaError_t value).
 */
#ifndef MOE_SYNTH_H
#define MOE_SYNTH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_synth_stream_t;

/* nblocks centred Q2_K blocks (84 B), from the random bytes r of the
 * stream: scale bytes 0..15 = sc | (3 sc) << 4 with sc = ((r & 15) * 6) >> 4
 * (min = 3 x scale), quants 16..79 = r, d = bytes 80, 81 with byte 81 =
 * (r & 3) | 0x18, dmin = d / 2 (byte 82 = byte 80, byte 83 = (r81 & 3) | 0x14):
 * each weight is d * sc * (q - 1.5). dst: device, 8-byte aligned. */
int moe_synth_q2k(void *dst, uint64_t nblocks, uint64_t key, moe_synth_stream_t stream);

/* nblocks random Q3_K blocks (110 B): random bytes, byte 109 (high byte of d)
 * forced to (b & 3) | 0x0C. */
int moe_synth_q3k(void *dst, uint64_t nblocks, uint64_t key, moe_synth_stream_t stream);

/* n bf16 values: the centred sum of the four 16-bit fields of word i times
 * `scale` (one f32 rounding), rounded to nearest-even bf16. */
int moe_synth_normal_bf16(uint16_t *dst, uint64_t n, uint64_t key, float scale, moe_synth_stream_t stream);

/* n f32 values lo + a * u, u = (word i >> 40) * 2^-24, two f32 roundings. */
int moe_synth_uniform_f32(float *dst, uint64_t n, uint64_t key, float lo, float a, moe_synth_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif
