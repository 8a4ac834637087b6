// gdn_umma.cuh -- 5th-generation tensor-core helpers (tcgen05, sm_100+): shared
// memory operand layout, descriptors, MMA issue, commit and TMEM access.
//
// Operands live in shared memory in the canonical no-swizzle layout: 8x8 bf16
// "core matrices" of 128 contiguous bytes (8 rows x 16 bytes).  A K-major
// operand of R rows x Ktot columns places element (r, k) at
//   (r/8)*(Ktot/8)*128 + (k/8)*128 + (r%8)*16 + (k%8)*2,
// so the descriptor's leading-dimension offset (next core matrix along K) is
// 128 bytes and its stride-dimension offset (next 8 rows) is (Ktot/8)*128.  The
// same bytes read as an MN-major operand (rows become K, columns become M) take
// LBO = (Ktot/8)*128 and SBO = 128.
//
// fp32 values enter the tensor core as bf16 hi/lo pairs (x = hi + lo + O(2^-16 x)):
// an operand stores its hi part at columns [0, K) and its lo part at [K, 2K), and
// a product accumulates hi*hi + hi*lo + lo*hi in fp32, which keeps about 16
// significant bits per operand instead of bf16's 8.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn_tma.cuh"

namespace gdn {
namespace umma {

__device__ __forceinline__ uint32_t kmajor_offset(int r, int k, int ktot) {
    return (uint32_t)((r >> 3) * (ktot >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}

// kind::f16 instruction descriptor: bf16 A and B, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major = false) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn_major ? (1u << 15) : 0u) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// D (+)= op(A) op(B) over K logical columns; A gives M rows, B gives N columns.
// A K-major operand is stored [M (or N) rows][2K]; an MN-major one is stored
// [K rows][2M (or 2N)], i.e. the same canonical layout read transposed (its
// leading-dimension offset then steps along K and its stride offset along M/N).
// Issued by one thread: descriptors are formed once and advanced by adding
// byte offsets / 16 to their address field.
__device__ __forceinline__ void mma_split(uint32_t d_tmem, const unsigned char* a, bool a_mn, const unsigned char* b,
                                          bool b_mn, int M, int N, int K, bool accumulate) {
    const uint32_t idesc = idesc_bf16(M, N, a_mn) | (b_mn ? (1u << 16) : 0u);
    const uint32_t a_row = (uint32_t)(2 * M / 8) * 128, b_row = (uint32_t)(2 * N / 8) * 128;
    const uint32_t k_row = (uint32_t)(2 * K / 8) * 128;
    const uint64_t da = a_mn ? smem_desc(smem_u32(a), a_row, 128) : smem_desc(smem_u32(a), 128, k_row);
    const uint64_t db = b_mn ? smem_desc(smem_u32(b), b_row, 128) : smem_desc(smem_u32(b), 128, k_row);
    const uint64_t a_step = (a_mn ? 2 * a_row : 256) / 16, b_step = (b_mn ? 2 * b_row : 256) / 16;  // 16 along K
    const uint64_t a_lo = (uint64_t)((a_mn ? M : K) / 8) * 128 / 16, b_lo = (uint64_t)((b_mn ? N : K) / 8) * 128 / 16;
    bool acc = accumulate;
    for (int ks = 0; ks < K / 16; ++ks) {
        const uint64_t ka = da + ks * a_step, kb = db + ks * b_step;
        mma_bf16(d_tmem, ka, kb, idesc, acc);            // hi * hi
        mma_bf16(d_tmem, ka, kb + b_lo, idesc, true);    // hi * lo
        mma_bf16(d_tmem, ka + a_lo, kb, idesc, true);    // lo * hi
        acc = true;
    }
}

// The same product when B is MN-major with its hi and lo halves side by side
// ([K rows][2N], hi in columns 0..N-1): per k-step one MMA of width 2N gives
// [A_hi B_hi | A_hi B_lo] and one of width N adds A_lo B_hi to the first half, so
// the product is D[:, 0:N] + D[:, N:2N] -- two instructions per k-step instead of
// three.  D takes 2N TMEM columns.
__device__ __forceinline__ void mma_split_bpair(uint32_t d_tmem, const unsigned char* a, bool a_mn, const unsigned char* b,
                                                int M, int N, int K, bool accumulate) {
    const uint32_t idesc2 = idesc_bf16(M, 2 * N, a_mn) | (1u << 16), idesc1 = idesc_bf16(M, N, a_mn) | (1u << 16);
    const uint32_t a_row = (uint32_t)(2 * M / 8) * 128, b_row = (uint32_t)(2 * N / 8) * 128;
    const uint32_t k_row = (uint32_t)(2 * K / 8) * 128;
    const uint64_t da = a_mn ? smem_desc(smem_u32(a), a_row, 128) : smem_desc(smem_u32(a), 128, k_row);
    const uint64_t db = smem_desc(smem_u32(b), b_row, 128);
    const uint64_t a_step = (a_mn ? 2 * a_row : 256) / 16, b_step = 2 * b_row / 16;  // 16 along K
    const uint64_t a_lo = (uint64_t)((a_mn ? M : K) / 8) * 128 / 16;
    bool acc = accumulate;
    for (int ks = 0; ks < K / 16; ++ks) {
        const uint64_t ka = da + ks * a_step, kb = db + ks * b_step;
        mma_bf16(d_tmem, ka, kb, idesc2, acc);          // hi * [hi | lo]
        mma_bf16(d_tmem, ka + a_lo, kb, idesc1, true);  // lo * hi
        acc = true;
    }
}

// Store 8 consecutive fp32 values as the hi and lo halves of row r, columns
// c0..c0+7 (c0 % 8 == 0) of a split operand image with N logical columns:
// two 16-byte stores.
__device__ __forceinline__ void store_split8(unsigned char* base, int r, int c0, int N, const float* v) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        const float2 hf = __bfloat1622float2(h2);
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(v[2 * j] - hf.x, v[2 * j + 1] - hf.y);
        hi[j] = *reinterpret_cast<const uint32_t*>(&h2);
        lo[j] = *reinterpret_cast<const uint32_t*>(&l2);
    }
    *reinterpret_cast<uint4*>(base + kmajor_offset(r, c0, 2 * N)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(base + kmajor_offset(r, N + c0, 2 * N)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

__device__ __forceinline__ void commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// One warp: allocate ncols TMEM columns (power of two >= 32); the address lands in *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 consecutive fp32 columns of TMEM lane (warp's sub-partition base + lane id).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

}  // namespace umma
}  // namespace gdn
