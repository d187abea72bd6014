// moe_synth.cu -- device twin of the seeded input generator (synth.py); see
// include/moe_synth.h. Pure integer work plus single IEEE-rounded f32
// operations, so every byte equals the host generator's.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_synth.h"

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t word(uint64_t key, uint64_t i)
{
    uint64_t z = key + (i + 1) * kGolden;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// random bytes with two byte positions per block remapped to (b & 3) | fix
__global__ void kblocks_kernel(uint8_t *dst, uint64_t nbytes, uint64_t key, uint32_t block, uint32_t pos_a,
                               uint32_t pos_b, uint32_t fix)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t w = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; w * 8 < nbytes; w += stride) {
        uint64_t v = word(key, w);
        const uint64_t p0 = w * 8;
        uint32_t off = (uint32_t)(p0 % block);
        uint8_t b[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint8_t x = (uint8_t)(v >> (8 * j));
            if (off == pos_a || off == pos_b)
                x = (uint8_t)((x & 3u) | fix);
            b[j] = x;
            off = off + 1 == block ? 0 : off + 1;
        }
        if (p0 + 8 <= nbytes) {
            uint64_t o = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                o |= (uint64_t)b[j] << (8 * j);
            *reinterpret_cast<uint64_t *>(dst + p0) = o;
        } else {
            for (int j = 0; p0 + j < nbytes; ++j)
                dst[p0 + j] = b[j];
        }
    }
}

__device__ __forceinline__ uint32_t rbyte(uint64_t key, uint64_t pos)
{
    return (uint32_t)(word(key, pos >> 3) >> (8 * (pos & 7))) & 0xFFu;
}

// centred Q2_K blocks (see moe_synth_q2k): one thread per 8 bytes
__global__ void q2k_kernel(uint8_t *dst, uint64_t nbytes, uint64_t key)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t w = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; w * 8 < nbytes; w += stride) {
        const uint64_t p0 = w * 8;
        uint8_t b[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint64_t p = p0 + j;
            const uint32_t off = (uint32_t)(p % 84);
            const uint32_t r = rbyte(key, p);
            uint32_t v = r;
            if (off < 16) {
                const uint32_t sc = ((r & 0x0Fu) * 6u) >> 4;
                v = sc | ((3u * sc) << 4);
            } else if (off == 81) {
                v = (r & 3u) | 0x18u;
            } else if (off == 82) {
                v = rbyte(key, p - 2);
            } else if (off == 83) {
                v = (rbyte(key, p - 2) & 3u) | 0x14u;
            }
            b[j] = (uint8_t)v;
        }
        if (p0 + 8 <= nbytes) {
            uint64_t o = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                o |= (uint64_t)b[j] << (8 * j);
            *reinterpret_cast<uint64_t *>(dst + p0) = o;
        } else {
            for (int j = 0; p0 + j < nbytes; ++j)
                dst[p0 + j] = b[j];
        }
    }
}

__global__ void normal_bf16_kernel(uint16_t *dst, uint64_t n, uint64_t key, float scale)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint64_t w = word(key, i);
        const int s = (int)(w & 0xFFFF) + (int)((w >> 16) & 0xFFFF) + (int)((w >> 32) & 0xFFFF) + (int)(w >> 48);
        const float f = __fmul_rn((float)(s - 131070), scale);
        const uint32_t b = __float_as_uint(f);
        dst[i] = (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
    }
}

__global__ void uniform_f32_kernel(float *dst, uint64_t n, uint64_t key, float lo, float a)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const float u = __fmul_rn((float)(uint32_t)(word(key, i) >> 40), 0x1p-24f);
        dst[i] = __fadd_rn(__fmul_rn(u, a), lo);
    }
}

int grid_for(uint64_t items)
{
    uint64_t g = (items + 255) / 256;
    return (int)(g < 8192 ? (g ? g : 1) : 8192);
}

}  // namespace

extern "C" {

int moe_synth_q2k(void *dst, uint64_t nblocks, uint64_t key, moe_synth_stream_t stream)
{
    const uint64_t nb = nblocks * 84;
    q2k_kernel<<<grid_for((nb + 7) / 8), 256, 0, (cudaStream_t)stream>>>(static_cast<uint8_t *>(dst), nb, key);
    return (int)cudaGetLastError();
}

int moe_synth_q3k(void *dst, uint64_t nblocks, uint64_t key, moe_synth_stream_t stream)
{
    const uint64_t nb = nblocks * 110;
    kblocks_kernel<<<grid_for((nb + 7) / 8), 256, 0, (cudaStream_t)stream>>>(static_cast<uint8_t *>(dst), nb, key,
                                                                            110, 109, 109, 0x0C);
    return (int)cudaGetLastError();
}

int moe_synth_normal_bf16(uint16_t *dst, uint64_t n, uint64_t key, float scale, moe_synth_stream_t stream)
{
    normal_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(dst, n, key, scale);
    return (int)cudaGetLastError();
}

int moe_synth_uniform_f32(float *dst, uint64_t n, uint64_t key, float lo, float a, moe_synth_stream_t stream)
{
    uniform_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(dst, n, key, lo, a);
    return (int)cudaGetLastError();
}

}  // extern "C"
