// Helpers shared by the tcgen05 prefill kernels: tensor-memory row loads and
// P stores, shared-memory operand descriptors for 128-byte-swizzled tiles, and
// paired fp32 arithmetic (f32x2) of sm_100-class SMs.
#pragma once

#include "ptx_sm103.cuh"

namespace attn {
namespace tc {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kErrWait = 0x8u;
constexpr unsigned kErrSeqlens = 0x10u;  // a packed batch gave an invalid sequence span
constexpr int kHalfRowBytes = 128;  // one D half (64 bf16) per shared-memory row

// Ties a register array to the preceding tcgen05.wait so that no use of the
// loaded values is scheduled before the wait.
ATTN_DEV void reg_dep(uint32_t (&r)[32]) {
    asm volatile("" : ATTN_P8(0), ATTN_P8(8), ATTN_P8(16), ATTN_P8(24) : : "memory");
}
ATTN_DEV void reg_dep(uint32_t (&r)[16]) {
    asm volatile("" : ATTN_P8(0), ATTN_P8(8) : : "memory");
}

// Loads N (multiple of 16) fp32 columns of this thread's TMEM lane.
template <int N>
ATTN_DEV void tmem_load_row(uint32_t taddr, float (&x)[N]) {
    uint32_t r[N / 32 > 0 ? N / 32 : 1][32];
    uint32_t t[16];
#pragma unroll
    for (int c = 0; c < N / 32; ++c) ptx::tmem_ld32(taddr + c * 32, r[c]);
    if constexpr (N % 32) ptx::tmem_ld16(taddr + (N / 32) * 32, t);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int c = 0; c < N / 32; ++c) {
        reg_dep(r[c]);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(r[c][i]);
    }
    if constexpr (N % 32) {
        reg_dep(t);
#pragma unroll
        for (int i = 0; i < 16; ++i) x[(N / 32) * 32 + i] = __uint_as_float(t[i]);
    }
}

// Writes P (N fp32 values) as N/2 packed bf16x2 columns at taddr.
template <int N>
ATTN_DEV void tmem_store_p(uint32_t taddr, const float (&p)[N]) {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = ptx::pack_bf16x2(p[c * 32 + 2 * i], p[c * 32 + 2 * i + 1]);
        ptx::tmem_st16(taddr + c * 16, r);
    }
    if constexpr (N % 32) {
        static_assert(N % 32 == 16, "N must be a multiple of 16");
        constexpr int base = (N / 32) * 32;
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                taddr + base / 2),
            "r"(ptx::pack_bf16x2(p[base + 0], p[base + 1])),
            "r"(ptx::pack_bf16x2(p[base + 2], p[base + 3])),
            "r"(ptx::pack_bf16x2(p[base + 4], p[base + 5])),
            "r"(ptx::pack_bf16x2(p[base + 6], p[base + 7])),
            "r"(ptx::pack_bf16x2(p[base + 8], p[base + 9])),
            "r"(ptx::pack_bf16x2(p[base + 10], p[base + 11])),
            "r"(ptx::pack_bf16x2(p[base + 12], p[base + 13])),
            "r"(ptx::pack_bf16x2(p[base + 14], p[base + 15]))
            : "memory");
    }
}

// This thread's row of a 128-row bf16 tile held as two 128-byte-swizzled D
// halves (64 d each) -> 64 TMEM columns at taddr, d pairs in order: the A
// operand layout of a tcgen05.mma that reads A from TMEM.
ATTN_DEV void row_to_tmem(const uint8_t *half0, const uint8_t *half1, uint32_t taddr, int row) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {  // 32 d at a time
        const uint8_t *src = ((q4 >> 1) ? half1 : half0) + row * kHalfRowBytes;
        uint32_t r[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // logical 16-byte chunk c: d 8c .. 8c+7 of the half
            const int c = 4 * (q4 & 1) + j;
            const uint4 v = *reinterpret_cast<const uint4 *>(src + ((c ^ (row & 7)) << 4));
            r[4 * j + 0] = v.x;
            r[4 * j + 1] = v.y;
            r[4 * j + 2] = v.z;
            r[4 * j + 3] = v.w;
        }
        ptx::tmem_st16(taddr + 16 * q4, r);
    }
}

// K-major operand tile (rows of 128 B, 8-row groups 1024 B apart), advanced by
// kk 16-element steps inside the 128-byte swizzle span.
ATTN_DEV uint64_t kmajor_desc(const uint8_t *tile, int kk) {
    return ptx::sdesc_sw128(ptx::smem_u32(tile) + kk * 32, 16, 1024);
}
// MN-major V tile: 16 keys per step (2048 B), D halves `half_stride` apart.
ATTN_DEV uint64_t vmajor_desc(const uint8_t *tile, int kk, uint32_t half_stride) {
    return ptx::sdesc_sw128(ptx::smem_u32(tile) + kk * 2048, half_stride, 1024);
}

// ---- paired fp32 arithmetic (one instruction for two lanes of a pair)
ATTN_DEV uint64_t f2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
ATTN_DEV float2 f2_split(uint64_t r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
ATTN_DEV uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
ATTN_DEV uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
ATTN_DEV uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// max of three fp32 values in one instruction
ATTN_DEV float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

}  // namespace tc
}  // namespace attn
