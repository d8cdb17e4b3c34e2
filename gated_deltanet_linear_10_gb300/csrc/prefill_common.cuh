// Device helpers shared by the tensor-core prefill kernels (internal header).
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace gdn {
namespace ptc {
using namespace tc;

constexpr int C = 64;                            // chunk
constexpr int DH = 128;                          // dk = dv
constexpr uint32_t kKQBytes = 2 * 128 * 128;     // 2 k-blocks x (64 K rows + 64 Q rows) x 128 B
constexpr uint32_t kKBlk = 128 * 128;            // k-block stride inside a K|Q stage
constexpr uint32_t kVBytes = 2 * 64 * 128;       // 2 k-blocks x 64 rows x 128 B
constexpr uint32_t kVBlk = 64 * 128;
constexpr uint32_t kMatBytes = 64 * 128;         // one 64 x 64 bf16 operand, one k-block
constexpr int kLd = 68;                          // fp32 row stride of the solve scratch
constexpr int kWbLd = 8;                         // row stride of a warp's 16 x 8 scratch
constexpr float kEps = 1e-6f;

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Rank -> sequence in decreasing-length order (ties by index), so that the
// longest chains start first.  Every thread tests a share of the candidates.
__device__ inline int seq_for_rank(const int32_t *cu, int n_seqs, int rank, int *slot) {
    if (n_seqs > 1024) return rank;
    if (threadIdx.x == 0) *slot = -1;
    __syncthreads();
    for (int i = threadIdx.x; i < n_seqs; i += blockDim.x) {
        const int li = cu[i + 1] - cu[i];
        int r = 0;
        for (int j = 0; j < n_seqs; ++j) {
            const int lj = cu[j + 1] - cu[j];
            r += (lj > li) || (lj == li && j < i);
        }
        if (r == rank) *slot = i;
    }
    __syncthreads();
    return *slot < 0 ? rank : *slot;
}

// Packed fp32 pairs (sm_100 and later): one instruction rounds each lane as
// its scalar counterpart does, so results equal the scalar code's.
__device__ __forceinline__ uint64_t f2_make(float a, float b) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ void f2_split(uint64_t d, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(d));
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Blocked UT solve helpers.  The 64 x 64 matrices are 4 x 4 blocks of 16.
// A warp computes half a block (16 rows x 8 columns): lane (r = lane/2,
// cg = lane%2) owns row r, columns col + 4cg .. col + 4cg + 3.
//   acc += X[xr.., xc..] (16 x 16) * Y[yr.., col..]
__device__ __forceinline__ void half_mac(float (&acc)[4], const float *X, int xr, int xc,
                                         const float *Y, int yr, int col, int r, int cg) {
    float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;   // second accumulator set: shorter chains
#pragma unroll
    for (int kk = 0; kk < 16; kk += 2) {
        const float x0 = X[(xr + r) * kLd + xc + kk];
        const float x1 = X[(xr + r) * kLd + xc + kk + 1];
        const float4 y0 = *reinterpret_cast<const float4 *>(Y + (yr + kk) * kLd + col + 4 * cg);
        const float4 y1 = *reinterpret_cast<const float4 *>(Y + (yr + kk + 1) * kLd + col + 4 * cg);
        acc[0] = fmaf(x0, y0.x, acc[0]);
        acc[1] = fmaf(x0, y0.y, acc[1]);
        acc[2] = fmaf(x0, y0.z, acc[2]);
        acc[3] = fmaf(x0, y0.w, acc[3]);
        e0 = fmaf(x1, y1.x, e0);
        e1 = fmaf(x1, y1.y, e1);
        e2 = fmaf(x1, y1.z, e2);
        e3 = fmaf(x1, y1.w, e3);
    }
    acc[0] += e0;
    acc[1] += e1;
    acc[2] += e2;
    acc[3] += e3;
}
// Tf[bi block rows][col..] = -Tf[bi][bi] * W, with W = acc (16 x 8) staged in wb.
__device__ __forceinline__ void half_finish(const float (&acc)[4], float *Tf, float *wb, int bi,
                                            int col, int r, int cg) {
    *reinterpret_cast<float4 *>(wb + r * kWbLd + 4 * cg) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    __syncwarp();
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f, p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
    for (int kk = 0; kk < 16; kk += 2) {
        const float d0 = Tf[(16 * bi + r) * kLd + 16 * bi + kk];
        const float d1 = Tf[(16 * bi + r) * kLd + 16 * bi + kk + 1];
        const float4 w0 = *reinterpret_cast<const float4 *>(wb + kk * kWbLd + 4 * cg);
        const float4 w1 = *reinterpret_cast<const float4 *>(wb + (kk + 1) * kWbLd + 4 * cg);
        o0 = fmaf(d0, w0.x, o0);
        o1 = fmaf(d0, w0.y, o1);
        o2 = fmaf(d0, w0.z, o2);
        o3 = fmaf(d0, w0.w, o3);
        p0 = fmaf(d1, w1.x, p0);
        p1 = fmaf(d1, w1.y, p1);
        p2 = fmaf(d1, w1.z, p2);
        p3 = fmaf(d1, w1.w, p3);
    }
    *reinterpret_cast<float4 *>(Tf + (16 * bi + r) * kLd + col + 4 * cg) =
        make_float4(-(o0 + p0), -(o1 + p1), -(o2 + p2), -(o3 + p3));
    __syncwarp();
}

__device__ __forceinline__ uint4 scale_chunk(uint4 w, float f) {
    uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 v = unpack_bf16(ws[e]);
        ws[e] = pack_bf16(v.x * f, v.y * f);
    }
    return make_uint4(ws[0], ws[1], ws[2], ws[3]);
}

// ---------------------------------------------------------------- prep --
// The state-independent part of a chunk, shared by the fused kernel and the
// chunk-parallel prep kernel.  256 "prep" threads (t = 0..255, 8 warps pw).

// Inverse L2 norm of row t / 2 of a raw K|Q stage (rows 0..63 K, 64..127 Q):
// threads t and t ^ 1 each sum one k-block and share the result.
__device__ __forceinline__ float kq_row_inv_norm(const uint8_t *kq, int t, int l2norm) {
    const uint32_t row = (uint32_t)(t >> 1), kb = (uint32_t)(t & 1);
    float ss = 0.f;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4 *>(kq + kb * kKBlk + sw128_chunk(row, ch));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16(ws[e]);
            ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
        }
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    return l2norm ? rsqrtf(ss + kEps) : 1.f;
}

// One row p of G = [K;Q] K^T, columns 32 chalf .. 32 chalf + 31, to
//   A_ij = beta_i D_ij r_k,i r_k,j G_ij    (K rows, j < i; fp32 into Af)
//   P_ij = scale D_ij r_q,i r_k,j G_ij     (Q rows, j <= i; bf16 into pdst)
// with D_ij = exp(gc_i - gc_j), walked downwards as a running product of
// alpha = exp(g): D_ii = 1, D_i,j-1 = D_ij alpha_j (one exp per row).
__device__ __forceinline__ void g_to_a_p(const uint32_t (&gr)[32], int p, int chalf, int n,
                                         const float *beta, const float *gam, const float *alpha,
                                         const float *rk, const float *rq, float scale, float *Af,
                                         uint8_t *pdst) {
    const bool krow = p < C;
    const int i = krow ? p : p - C;
    const bool ok = i < n;
    const int cb = 32 * chalf;
    const float coef = krow ? beta[i] * rk[i] : scale * rq[i];
    float e = (i > cb + 31) ? __expf(gam[i] - gam[cb + 31]) : 1.f;
    const int lim = ok ? (krow ? i : i + 1) : 0;      // kept: j < lim
    float rkc[32], alc[32];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float4 a4 = *reinterpret_cast<const float4 *>(rk + cb + 4 * q);
        const float4 b4 = *reinterpret_cast<const float4 *>(alpha + cb + 4 * q);
        rkc[4 * q] = a4.x; rkc[4 * q + 1] = a4.y; rkc[4 * q + 2] = a4.z; rkc[4 * q + 3] = a4.w;
        alc[4 * q] = b4.x; alc[4 * q + 1] = b4.y; alc[4 * q + 2] = b4.z; alc[4 * q + 3] = b4.w;
    }
    float v[32];
#pragma unroll
    for (int jj = 31; jj >= 0; --jj) {
        const int j = cb + jj;
        v[jj] = j < lim ? coef * e * rkc[jj] * __uint_as_float(gr[jj]) : 0.f;
        if (j <= i) e *= alc[jj];
    }
    if (krow) {
        float *arow = Af + i * kLd + cb;
#pragma unroll
        for (int jj = 0; jj < 32; jj += 4)
            *reinterpret_cast<float4 *>(arow + jj) = make_float4(v[jj], v[jj + 1], v[jj + 2], v[jj + 3]);
    } else {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t w[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) w[e2] = pack_bf16(v[cc * 8 + 2 * e2], v[cc * 8 + 2 * e2 + 1]);
            *reinterpret_cast<uint4 *>(pdst + sw128_chunk(i, 4 * chalf + cc)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// The four diagonal 16 x 16 blocks of T = (I + A)^-1 by forward
// substitution, exact fp32, on warps 0 and 1 of the 256 prep threads: lane c
// of half-warp hw solves column c of block 2 pw + hw,
//   T[r][c] = delta_rc - sum_{m < r} A[r][m] T[m][c]   (m ascending),
// reading the rows of A as broadcasts.  (One lane per row half, with the
// finished rows passed on by shuffles, took 8 shuffles per step on 4 warps.)
__device__ __forceinline__ void ut_diag_blocks(const float *Af, float *Tf, int pw, int lane) {
    if (pw >= 2) return;
    const int bb = 2 * pw + (lane >> 4), c = lane & 15;
    const float *Ab = Af + (16 * bb) * kLd + 16 * bb;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        float acc = r == c ? 1.f : 0.f;
#pragma unroll
        for (int m4 = 0; m4 < r; m4 += 4) {
            const float4 f = *reinterpret_cast<const float4 *>(Ab + r * kLd + m4);
            const float ar[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (m4 + u < r) acc = fmaf(-ar[u], x[m4 + u], acc);
        }
        x[r] = acc;
        // a compiler barrier: each row's loads stay next to their use
        // (hoisting all of them spills registers at the prep kernel's 72)
        asm volatile("" ::: "memory");
    }
    float *Tb = Tf + (16 * bb) * kLd + 16 * bb + c;
#pragma unroll
    for (int r = 0; r < 16; ++r) Tb[r * kLd] = x[r];
}

// T = (I + A)^-1 for the strictly lower triangular A in Af (fp32, row stride
// kLd), then T1 = T diag(beta) and (kT2) T2 = -T diag(beta xs) as bf16
// K-major operands at dst and dst + kMatBytes (xs = Gam r_k, zero on padded
// rows).
// The diagonal 16 x 16 blocks by forward substitution, then the blocks below
// the diagonal level by level (T_ij = -T_ii sum_k A_ik T_kj); Wb holds each
// warp's 16 x 8 scratch followed by a 16 x 16 partial sum.  Ends with the
// T1 / T2 writes issued (no barrier after the last of them).
template <bool kT2>
__device__ __forceinline__ void ut_solve(const float *Af, float *Tf, float *Wb, int t, int pw,
                                         int lane, const float *beta, const float *xs,
                                         uint8_t *dst) {
    float *Zs = Wb + 8 * 16 * kWbLd;
    ut_diag_blocks(Af, Tf, pw, lane);
    named_sync(1, 256);
    const int r = lane >> 1, cg = lane & 1;
    float *wb = Wb + pw * 16 * kWbLd;
    float acc[4];
    if (pw < 6) {              // level 1: T10, T21, T32
        const int b0 = pw >> 1, half = pw & 1;
        const int col = 16 * b0 + 8 * half;
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        half_mac(acc, Af, 16 * (b0 + 1), 16 * b0, Tf, 16 * b0, col, r, cg);
        half_finish(acc, Tf, wb, b0 + 1, col, r, cg);
    }
    named_sync(1, 256);
    if (pw < 6) {              // level 2: T20, T31 and Z30 = A30 T00 + A31 T10
        const int item = pw >> 1, half = pw & 1;
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        if (item == 0) {
            const int col = 8 * half;
            half_mac(acc, Af, 32, 0, Tf, 0, col, r, cg);
            half_mac(acc, Af, 32, 16, Tf, 16, col, r, cg);
            half_finish(acc, Tf, wb, 2, col, r, cg);
        } else if (item == 1) {
            const int col = 16 + 8 * half;
            half_mac(acc, Af, 48, 16, Tf, 16, col, r, cg);
            half_mac(acc, Af, 48, 32, Tf, 32, col, r, cg);
            half_finish(acc, Tf, wb, 3, col, r, cg);
        } else {
            const int col = 8 * half;
            half_mac(acc, Af, 48, 0, Tf, 0, col, r, cg);
            half_mac(acc, Af, 48, 16, Tf, 16, col, r, cg);
            *reinterpret_cast<float4 *>(Zs + r * 16 + col + 4 * cg) =
                make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
    }
    named_sync(1, 256);
    // block rows 0..2 are final now, block row 3 after level 3
    auto write_t12 = [&](int i, int ch) {
        uint32_t w1[4], w2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j0 = ch * 8 + 2 * e, j1 = j0 + 1;
            const float t0 = j0 <= i ? Tf[i * kLd + j0] : 0.f;
            const float t1 = j1 <= i ? Tf[i * kLd + j1] : 0.f;
            w1[e] = pack_bf16(t0 * beta[j0], t1 * beta[j1]);
            if (kT2) w2[e] = pack_bf16(-t0 * beta[j0] * xs[j0], -t1 * beta[j1] * xs[j1]);
        }
        *reinterpret_cast<uint4 *>(dst + sw128_chunk(i, ch)) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
        if (kT2)
            *reinterpret_cast<uint4 *>(dst + kMatBytes + sw128_chunk(i, ch)) =
                make_uint4(w2[0], w2[1], w2[2], w2[3]);
    };
    if (pw < 2) {              // level 3: T30 = -T33 (Z30 + A32 T20)
        const int col = 8 * pw;
        const float4 z = *reinterpret_cast<const float4 *>(Zs + r * 16 + col + 4 * cg);
        acc[0] = z.x; acc[1] = z.y; acc[2] = z.z; acc[3] = z.w;
        half_mac(acc, Af, 48, 32, Tf, 32, col, r, cg);
        half_finish(acc, Tf, wb, 3, col, r, cg);
    } else {                   // meanwhile rows 0..47: 384 chunks over 192 threads
        const int u = t - 64;
        write_t12(u >> 2, 2 * (u & 3));
        write_t12(u >> 2, 2 * (u & 3) + 1);
    }
    named_sync(1, 256);
    if (t < 128) write_t12(48 + (t >> 3), t & 7);
}

// ------------------------------------------- UT solve, block products on
// the warp-level tensor cores (mma.sync m16n8k8, tf32 in, fp32 accumulate).
// The 16 x 16 blocks are below the 64-row minimum of tcgen05, and each warp
// only ever needs a 16 x 8 half-block.  Fragment layouts (g = lane / 4,
// t = lane % 4): A 16 x 8 row-major a0 = A[g][t], a1 = A[g+8][t],
// a2 = A[g][t+4], a3 = A[g+8][t+4]; B 8 x 8 b0 = B[t][g], b1 = B[t+4][g];
// C 16 x 8 c0 = C[g][2t], c1 = C[g][2t+1], c2 = C[g+8][2t], c3 = C[g+8][2t+1].
__device__ __forceinline__ uint32_t tf32_of(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// acc += X[xr.., xc..] (16 x 16) * Y[yr.., col..col+7] (16 x 8); row stride kLd
__device__ __forceinline__ void hm_mac(float (&acc)[4], const float *X, int xr, int xc,
                                       const float *Y, int yr, int col, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 16; ks += 8) {
        const uint32_t a[4] = {tf32_of(X[(xr + g) * kLd + xc + ks + t]),
                               tf32_of(X[(xr + g + 8) * kLd + xc + ks + t]),
                               tf32_of(X[(xr + g) * kLd + xc + ks + t + 4]),
                               tf32_of(X[(xr + g + 8) * kLd + xc + ks + t + 4])};
        mma_tf32(acc, a, tf32_of(Y[(yr + ks + t) * kLd + col + g]),
                 tf32_of(Y[(yr + ks + t + 4) * kLd + col + g]));
    }
}
// Tf[block row bi][col..col+7] = -T_ii * W, W = acc (16 x 8) staged in wb
// (16 x 8 floats, this warp's own)
__device__ __forceinline__ void hm_finish(const float (&acc)[4], float *Tf, float *wb, int bi,
                                          int col, int lane) {
    const int g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2 *>(wb + g * 8 + 2 * t) = make_float2(acc[0], acc[1]);
    *reinterpret_cast<float2 *>(wb + (g + 8) * 8 + 2 * t) = make_float2(acc[2], acc[3]);
    __syncwarp();
    float out[4] = {0.f, 0.f, 0.f, 0.f};
    const float *Tii = Tf + 16 * bi * kLd + 16 * bi;
#pragma unroll
    for (int ks = 0; ks < 16; ks += 8) {
        const uint32_t a[4] = {tf32_of(-Tii[g * kLd + ks + t]), tf32_of(-Tii[(g + 8) * kLd + ks + t]),
                               tf32_of(-Tii[g * kLd + ks + t + 4]),
                               tf32_of(-Tii[(g + 8) * kLd + ks + t + 4])};
        mma_tf32(out, a, tf32_of(wb[(ks + t) * 8 + g]), tf32_of(wb[(ks + t + 4) * 8 + g]));
    }
    float *dst = Tf + (16 * bi) * kLd + col;
    *reinterpret_cast<float2 *>(dst + g * kLd + 2 * t) = make_float2(out[0], out[1]);
    *reinterpret_cast<float2 *>(dst + (g + 8) * kLd + 2 * t) = make_float2(out[2], out[3]);
    __syncwarp();
}

// acc += (neg ? -X : X) (16 x 16, row stride ldx) * Y (16 x 8, row stride ldy),
// tf32 operands, X and Y pointing at the blocks' first elements.
__device__ __forceinline__ void hm_mac_at(float (&acc)[4], const float *X, int ldx, const float *Y,
                                          int ldy, int lane, bool neg) {
    const int g = lane >> 2, t = lane & 3;
    const float sg = neg ? -1.f : 1.f;
#pragma unroll
    for (int ks = 0; ks < 16; ks += 8) {
        const uint32_t a[4] = {tf32_of(sg * X[g * ldx + ks + t]),
                               tf32_of(sg * X[(g + 8) * ldx + ks + t]),
                               tf32_of(sg * X[g * ldx + ks + t + 4]),
                               tf32_of(sg * X[(g + 8) * ldx + ks + t + 4])};
        mma_tf32(acc, a, tf32_of(Y[(ks + t) * ldy + g]), tf32_of(Y[(ks + t + 4) * ldy + g]));
    }
}

// ut_solve with the off-diagonal blocks on mma.sync (tf32 in, fp32
// accumulate), by the 2 x 2 block inverse at the 32-row level: with
// T_hi = (I + A_hi)^-1 over block rows 0, 1 and T_lo over rows 2, 3,
//   T10 = -T11 (A10 T00),  T32 = -T33 (A32 T22),
//   X = A_ll T_hi:  X20 = A20 T00 + A21 T10, X21 = A21 T11,
//                   X30 = A30 T00 + A31 T10, X31 = A31 T11,
//   [T20 T21; T30 T31] = -T_lo X:  T2j = -T22 X2j,  T3j = -(T32 X2j + T33 X3j).
// Three dependent stages of at most two 16 x 16 products each, where the
// block-row-by-block-row form chains six products from T10 to T30: stage 1
// T10, T32 (warps 0..3) and the parts of X that need no T10 (warps 4..7, kept
// in registers); stage 2 X20, X30 (warps 4..7), X into Wb, and the T1 / T2
// rows 0..31 (warps 0..3); stage 3 the lower-left quarter (one 16 x 8
// half-block per warp).  T20 and T21 come out as in the row form (-T22 times
// the same sums); T30 and T31 are associated differently.
template <bool kT2>
__device__ __forceinline__ void ut_solve_mma(const float *Af, float *Tf, float *Wb, int t, int pw,
                                             int lane, const float *beta, const float *xs,
                                             uint8_t *dst) {
    constexpr int kXLd = 36;                  // X: 32 x 32 fp32 in Wb
    static_assert(32 * kXLd <= 8 * 16 * kWbLd + 16 * 16, "X fits in the solve scratch");
    float *Xs = Wb;
    ut_diag_blocks(Af, Tf, pw, lane);
    named_sync(1, 256);
    const int g = lane >> 2, tq = lane & 3;
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
    const int h = pw & 1;                     // which 8 columns of a 16-column block
    if (pw < 4) {              // stage 1: T10 (warps 0, 1), T32 (warps 2, 3)
        const int bi = pw < 2 ? 1 : 3;        // block row; block column bi - 1
        const int col = 16 * (bi - 1) + 8 * h;
        hm_mac(acc, Af, 16 * bi, 16 * (bi - 1), Tf, 16 * (bi - 1), col, lane);
        hm_finish(acc, Tf, Wb + pw * 16 * kWbLd, bi, col, lane);
    } else {                   // X_r0 partial = A_r0 T00 and X_r1 = A_r1 T11 (r = 2 or 3)
        const int r = pw < 6 ? 2 : 3;
        hm_mac(acc, Af, 16 * r, 0, Tf, 0, 8 * h, lane);
        hm_mac(acc2, Af, 16 * r, 16, Tf, 16, 16 + 8 * h, lane);
    }
    named_sync(1, 256);
    auto write_t12 = [&](int i, int ch) {   // 8 columns: float4 loads of T, beta, xs
        float tv[8], bv[8], xv[8];
#pragma unroll
        for (int h4 = 0; h4 < 2; ++h4) {
            const float4 t4 = *reinterpret_cast<const float4 *>(Tf + i * kLd + ch * 8 + 4 * h4);
            const float4 b4 = *reinterpret_cast<const float4 *>(beta + ch * 8 + 4 * h4);
            tv[4 * h4] = t4.x; tv[4 * h4 + 1] = t4.y; tv[4 * h4 + 2] = t4.z; tv[4 * h4 + 3] = t4.w;
            bv[4 * h4] = b4.x; bv[4 * h4 + 1] = b4.y; bv[4 * h4 + 2] = b4.z; bv[4 * h4 + 3] = b4.w;
            if (kT2) {
                const float4 x4 = *reinterpret_cast<const float4 *>(xs + ch * 8 + 4 * h4);
                xv[4 * h4] = x4.x; xv[4 * h4 + 1] = x4.y; xv[4 * h4 + 2] = x4.z; xv[4 * h4 + 3] = x4.w;
            }
        }
        uint32_t w1[4], w2[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const float t0 = ch * 8 + e <= i ? tv[e] * bv[e] : 0.f;      // above the
            const float t1 = ch * 8 + e + 1 <= i ? tv[e + 1] * bv[e + 1] : 0.f;   // diagonal: 0
            w1[e / 2] = pack_bf16(t0, t1);
            if (kT2) w2[e / 2] = pack_bf16(-t0 * xv[e], -t1 * xv[e + 1]);
        }
        *reinterpret_cast<uint4 *>(dst + sw128_chunk(i, ch)) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
        if (kT2)
            *reinterpret_cast<uint4 *>(dst + kMatBytes + sw128_chunk(i, ch)) =
                make_uint4(w2[0], w2[1], w2[2], w2[3]);
    };
    if (pw >= 4) {             // stage 2: X_r0 += A_r1 T10, then X into Wb
        const int r = pw < 6 ? 2 : 3;
        hm_mac(acc, Af, 16 * r, 16, Tf, 16, 8 * h, lane);
        float *x0 = Xs + (16 * (r - 2)) * kXLd + 8 * h;        // X_r0, this half
        float *x1 = x0 + 16;                                    // X_r1
        *reinterpret_cast<float2 *>(x0 + g * kXLd + 2 * tq) = make_float2(acc[0], acc[1]);
        *reinterpret_cast<float2 *>(x0 + (g + 8) * kXLd + 2 * tq) = make_float2(acc[2], acc[3]);
        *reinterpret_cast<float2 *>(x1 + g * kXLd + 2 * tq) = make_float2(acc2[0], acc2[1]);
        *reinterpret_cast<float2 *>(x1 + (g + 8) * kXLd + 2 * tq) = make_float2(acc2[2], acc2[3]);
    } else {                   // meanwhile T1 / T2 rows 0..31 (block rows 0, 1 are final)
        write_t12(t >> 2, 2 * (t & 3));
        write_t12(t >> 2, 2 * (t & 3) + 1);
    }
    named_sync(1, 256);
    {                          // stage 3: warp pw -> block (2 + pw / 4, (pw / 2) % 2), half h
        const int r = 2 + (pw >> 2), cb = (pw >> 1) & 1;
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        const float *xr = Xs + cb * 16 + 8 * h;                // X_2cb, this half
        if (r == 2) {          // T2cb = -T22 X2cb
            hm_mac_at(o, Tf + 32 * kLd + 32, kLd, xr, kXLd, lane, true);
        } else {               // T3cb = -(T32 X2cb + T33 X3cb)
            hm_mac_at(o, Tf + 48 * kLd + 32, kLd, xr, kXLd, lane, true);
            hm_mac_at(o, Tf + 48 * kLd + 48, kLd, xr + 16 * kXLd, kXLd, lane, true);
        }
        float *dstT = Tf + (16 * r) * kLd + 16 * cb + 8 * h;
        *reinterpret_cast<float2 *>(dstT + g * kLd + 2 * tq) = make_float2(o[0], o[1]);
        *reinterpret_cast<float2 *>(dstT + (g + 8) * kLd + 2 * tq) = make_float2(o[2], o[3]);
    }
    named_sync(1, 256);
    write_t12(32 + (t >> 3), t & 7);
}

}  // namespace ptc
}  // namespace gdn
