// attention.cu -- causal multi-head attention forward/backward (sm_103a).
//
// Computes, per (b, h), S = Q K^T / sqrt(HS) with keys j <= query i,
// P = softmax(S), O = P V, saving only the per-row log-sum-exp (LSE) of S;
// the backward recomputes P from the LSE (flash-attention form of
// llm.c "train_gpt2.cu" attention_forward / attention_backward with
// softmax_forward_kernel5 and softmax_autoregressive_backward_kernel:
// dP = dO V^T, dS = P (dP - rowsum(dO o O)), dQ = dS K / sqrt(HS),
// dK = dS^T Q / sqrt(HS), dV = P^T dO).
// Q, K, V are read in place from the fused (B, T, 3, NH, HS) QKV activation;
// the output is written as (B, T, NH, HS). No (T x T) matrix is stored.
//
// Two implementations:
//  * SIMT (any head size <= 128; fp32 or bf16 storage): one thread per
//    query row (forward, dQ) or key row (dK, dV), fp32 online softmax.
//  * bf16 tensor-core flash kernels for head size 64: 64-row blocks, four
//    warps x 16 rows, m16n8k16 bf16 MMAs with fp32 accumulation, K/V tiles
//    double-buffered in XOR-swizzled shared memory via cp.async. The
//    backward is deterministic: one kernel owns dQ per query block, another
//    owns dK/dV per key block; nothing is accumulated with atomics.
#include "common.cuh"
#include "internal.h"

#include "gpt2.h"

namespace gk {

#define LOG2E_F 1.4426950408889634f
#define LN2_F 0.6931471805599453f

// ================================================================== SIMT
template <typename T, int HS>
__global__ void attn_fwd_simt_k(T* __restrict__ out, float* __restrict__ lse,
                                const T* __restrict__ qkv, int B, int Tn, int C, int NH) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= B * NH * Tn) return;
    const int i = idx % Tn, h = (idx / Tn) % NH, b = idx / (Tn * NH);
    const size_t C3 = 3 * (size_t)C;
    const T* q = qkv + ((size_t)b * Tn + i) * C3 + (size_t)h * HS;
    const float scale = rsqrtf((float)HS);
    float qr[HS], o[HS];
#pragma unroll
    for (int d = 0; d < HS; d++) {
        qr[d] = to_f(q[d]) * scale;
        o[d] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j <= i; j++) {
        const T* k = qkv + ((size_t)b * Tn + j) * C3 + C + (size_t)h * HS;
        const T* v = k + C;
        float s = 0.f;
#pragma unroll
        for (int d = 0; d < HS; d++) s += qr[d] * to_f(k[d]);
        const float mn = fmaxf(m, s);
        const float corr = expf(m - mn), p = expf(s - mn);
        l = l * corr + p;
#pragma unroll
        for (int d = 0; d < HS; d++) o[d] = o[d] * corr + p * to_f(v[d]);
        m = mn;
    }
    T* y = out + ((size_t)b * Tn + i) * C + (size_t)h * HS;
    const float inv = 1.f / l;
#pragma unroll
    for (int d = 0; d < HS; d++) y[d] = from_f<T>(o[d] * inv);
    lse[((size_t)b * NH + h) * Tn + i] = m + logf(l);
}

// D[b,h,i] = sum_d dO[b,i,h,d] O[b,i,h,d]
template <typename T>
__global__ void attn_rowdot_k(float* __restrict__ D, const T* __restrict__ dout,
                              const T* __restrict__ out, int B, int Tn, int C, int NH, int HS) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= B * NH * Tn) return;
    const int i = idx % Tn, h = (idx / Tn) % NH, b = idx / (Tn * NH);
    const size_t off = ((size_t)b * Tn + i) * C + (size_t)h * HS;
    float s = 0.f;
    for (int d = 0; d < HS; d++) s += to_f(dout[off + d]) * to_f(out[off + d]);
    D[idx] = s;
}

template <typename T, int HS>
__global__ void attn_bwd_dq_simt_k(T* __restrict__ dqkv, const T* __restrict__ dout,
                                   const T* __restrict__ qkv, const float* __restrict__ lse,
                                   const float* __restrict__ D, int B, int Tn, int C, int NH) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= B * NH * Tn) return;
    const int i = idx % Tn, h = (idx / Tn) % NH, b = idx / (Tn * NH);
    const size_t C3 = 3 * (size_t)C;
    const float scale = rsqrtf((float)HS);
    const T* q = qkv + ((size_t)b * Tn + i) * C3 + (size_t)h * HS;
    const T* dO = dout + ((size_t)b * Tn + i) * C + (size_t)h * HS;
    float qr[HS], dor[HS], dq[HS];
#pragma unroll
    for (int d = 0; d < HS; d++) {
        qr[d] = to_f(q[d]) * scale;
        dor[d] = to_f(dO[d]);
        dq[d] = 0.f;
    }
    const float li = lse[idx], Di = D[idx];
    for (int j = 0; j <= i; j++) {
        const T* k = qkv + ((size_t)b * Tn + j) * C3 + C + (size_t)h * HS;
        const T* v = k + C;
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < HS; d++) {
            s += qr[d] * to_f(k[d]);
            dp += dor[d] * to_f(v[d]);
        }
        const float ds = expf(s - li) * (dp - Di);
#pragma unroll
        for (int d = 0; d < HS; d++) dq[d] += ds * to_f(k[d]);
    }
    T* dst = dqkv + ((size_t)b * Tn + i) * C3 + (size_t)h * HS;
#pragma unroll
    for (int d = 0; d < HS; d++) dst[d] = from_f<T>(dq[d] * scale);
}

template <typename T, int HS>
__global__ void attn_bwd_dkv_simt_k(T* __restrict__ dqkv, const T* __restrict__ dout,
                                    const T* __restrict__ qkv, const float* __restrict__ lse,
                                    const float* __restrict__ D, int B, int Tn, int C, int NH) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= B * NH * Tn) return;
    const int j = idx % Tn, h = (idx / Tn) % NH, b = idx / (Tn * NH);
    const size_t C3 = 3 * (size_t)C;
    const float scale = rsqrtf((float)HS);
    const T* k = qkv + ((size_t)b * Tn + j) * C3 + C + (size_t)h * HS;
    const T* v = k + C;
    float kr[HS], vr[HS], dk[HS], dv[HS];
#pragma unroll
    for (int d = 0; d < HS; d++) {
        kr[d] = to_f(k[d]) * scale;
        vr[d] = to_f(v[d]);
        dk[d] = 0.f;
        dv[d] = 0.f;
    }
    const size_t row0 = ((size_t)b * NH + h) * Tn;
    for (int i = j; i < Tn; i++) {
        const T* q = qkv + ((size_t)b * Tn + i) * C3 + (size_t)h * HS;
        const T* dO = dout + ((size_t)b * Tn + i) * C + (size_t)h * HS;
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < HS; d++) {
            s += to_f(q[d]) * kr[d];
            dp += to_f(dO[d]) * vr[d];
        }
        const float p = expf(s - lse[row0 + i]);
        const float ds = p * (dp - D[row0 + i]);
#pragma unroll
        for (int d = 0; d < HS; d++) {
            dv[d] += p * to_f(dO[d]);
            dk[d] += ds * to_f(q[d]);
        }
    }
    T* dkp = dqkv + ((size_t)b * Tn + j) * C3 + C + (size_t)h * HS;
    T* dvp = dkp + C;
#pragma unroll
    for (int d = 0; d < HS; d++) {
        dkp[d] = from_f<T>(dk[d] * scale);
        dvp[d] = from_f<T>(dv[d]);
    }
}

// ================================================================== bf16 flash (HS = 64)
namespace fa {

constexpr int BLK = 64;  // rows per block (queries or keys)
constexpr int HSZ = 64;  // head size

DEVI uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// element offset of (row, 16-byte chunk) in a 64x64 bf16 tile with XOR swizzle
DEVI int swz(int row, int chunk) { return row * HSZ + ((chunk ^ (row & 7)) << 3); }

DEVI void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
DEVI void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> DEVI void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// load rows [r0, r0+64) of a (T, 64) head slice with row pitch `pitch`; rows >= Tn are zero
DEVI void load_tile(bf16* tile, const bf16* g, int r0, int Tn, size_t pitch) {
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int c = threadIdx.x + 128 * i;
        const int row = c >> 3, ch = c & 7;
        const bool valid = r0 + row < Tn;
        const bf16* src = valid ? g + (size_t)(r0 + row) * pitch + ch * 8 : g;
        cp_async16(saddr(tile + swz(row, ch)), src, valid);
    }
}

DEVI void ldsm4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
DEVI void ldsm4t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
DEVI void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
DEVI uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// A fragments (16 rows starting at row0, all 64 columns) of a swizzled tile
DEVI void load_a_frags(uint32_t (&f)[4][4], const bf16* tile, int row0) {
    const int lane = threadIdx.x & 31;
    const int row = row0 + (lane & 15);
#pragma unroll
    for (int kk = 0; kk < 4; kk++) ldsm4(f[kk], saddr(tile + swz(row, 2 * kk + (lane >> 4))));
}

// acc[16 x 64] += A(16 x 64, fragments) . Tile^T where Tile rows are the n index
// (B operand taken "col-major" straight from row-major rows: non-transposed ldmatrix)
DEVI void mma_abt(float (&acc)[8][4], const uint32_t (&a)[4][4], const bf16* tile) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int np = 0; np < 4; np++) {
        const int row = np * 16 + ((lane >> 4) << 3) + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < 4; kk++) {
            uint32_t r[4];
            ldsm4(r, saddr(tile + swz(row, 2 * kk + ((lane >> 3) & 1))));
            mma16816(acc[2 * np], a[kk], r[0], r[1]);
            mma16816(acc[2 * np + 1], a[kk], r[2], r[3]);
        }
    }
}

// acc[16 x 64] += P(16 x 64 over tile rows, as accumulator-layout floats) . Tile
// where Tile rows are the k index (transposed ldmatrix)
DEVI void mma_pv(float (&acc)[8][4], const float (&p)[8][4], const bf16* tile) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int kk = 0; kk < 4; kk++) {
        uint32_t a[4];
        a[0] = pack_bf16(p[2 * kk][0], p[2 * kk][1]);
        a[1] = pack_bf16(p[2 * kk][2], p[2 * kk][3]);
        a[2] = pack_bf16(p[2 * kk + 1][0], p[2 * kk + 1][1]);
        a[3] = pack_bf16(p[2 * kk + 1][2], p[2 * kk + 1][3]);
        const int row = kk * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
#pragma unroll
        for (int cp = 0; cp < 4; cp++) {
            uint32_t r[4];
            ldsm4t(r, saddr(tile + swz(row, 2 * cp + (lane >> 4))));
            mma16816(acc[2 * cp], a, r[0], r[1]);
            mma16816(acc[2 * cp + 1], a, r[2], r[3]);
        }
    }
}

DEVI void zero_acc(float (&a)[8][4]) {
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) a[i][j] = 0.f;
}

__global__ void __launch_bounds__(128) flash_fwd_k(bf16* __restrict__ out, float* __restrict__ lse,
                                                   const bf16* __restrict__ qkv, int Tn, int C,
                                                   int NH, float scale_log2) {
    __shared__ __align__(128) bf16 sQ[BLK * HSZ];
    __shared__ __align__(128) bf16 sK[2][BLK * HSZ];
    __shared__ __align__(128) bf16 sV[2][BLK * HSZ];
    const int qb = gridDim.x - 1 - blockIdx.x;  // heaviest (most keys) first
    const int b = blockIdx.y / NH, h = blockIdx.y % NH;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t pitch = 3 * (size_t)C;
    const bf16* Qg = qkv + (size_t)b * Tn * pitch + (size_t)h * HSZ;
    const bf16* Kg = Qg + C;
    const bf16* Vg = Qg + 2 * C;
    load_tile(sQ, Qg, qb * BLK, Tn, pitch);
    load_tile(sK[0], Kg, 0, Tn, pitch);
    load_tile(sV[0], Vg, 0, Tn, pitch);
    cp_commit();

    uint32_t qf[4][4];
    float o[8][4];
    zero_acc(o);
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    const int nkb = qb + 1;
    for (int kb = 0; kb < nkb; kb++) {
        if (kb + 1 < nkb) {
            load_tile(sK[(kb + 1) & 1], Kg, (kb + 1) * BLK, Tn, pitch);
            load_tile(sV[(kb + 1) & 1], Vg, (kb + 1) * BLK, Tn, pitch);
            cp_commit();
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        if (kb == 0) load_a_frags(qf, sQ, warp * 16);
        float s[8][4];
        zero_acc(s);
        mma_abt(s, qf, sK[kb & 1]);
        // scale into log2 units and apply the causal mask on the diagonal block
        const int qr = warp * 16 + (lane >> 2);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                float v = s[nt][e] * scale_log2;
                if (kb == qb) {
                    const int key = nt * 8 + 2 * (lane & 3) + (e & 1);
                    const int qrow = qr + ((e >> 1) << 3);
                    if (key > qrow) v = -INFINITY;
                }
                s[nt][e] = v;
            }
        }
#pragma unroll
        for (int r = 0; r < 2; r++) {
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; nt++) mx = fmaxf(mx, fmaxf(s[nt][2 * r], s[nt][2 * r + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mn = fmaxf(m[r], mx);
            const float corr = exp2f(m[r] - mn);
            float ls = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; nt++) {
                s[nt][2 * r] = exp2f(s[nt][2 * r] - mn);
                s[nt][2 * r + 1] = exp2f(s[nt][2 * r + 1] - mn);
                ls += s[nt][2 * r] + s[nt][2 * r + 1];
                o[nt][2 * r] *= corr;
                o[nt][2 * r + 1] *= corr;
            }
            l[r] = l[r] * corr + ls;
            m[r] = mn;
        }
        mma_pv(o, s, sV[kb & 1]);
        __syncthreads();
    }
    // finalise: quad-reduce the row sums, normalise, write O and the LSE
#pragma unroll
    for (int r = 0; r < 2; r++) {
        float lt = l[r];
        lt += __shfl_xor_sync(0xffffffffu, lt, 1);
        lt += __shfl_xor_sync(0xffffffffu, lt, 2);
        const int q = qb * BLK + warp * 16 + (lane >> 2) + 8 * r;
        if (q < Tn) {
            const float inv = 1.f / lt;
            bf16* y = out + ((size_t)b * Tn + q) * C + (size_t)h * HSZ;
#pragma unroll
            for (int nt = 0; nt < 8; nt++) {
                const int d = nt * 8 + 2 * (lane & 3);
                *reinterpret_cast<uint32_t*>(y + d) =
                    pack_bf16(o[nt][2 * r] * inv, o[nt][2 * r + 1] * inv);
            }
            if ((lane & 3) == 0) lse[((size_t)b * NH + h) * Tn + q] = (m[r] + log2f(lt)) * LN2_F;
        }
    }
}

// dQ for one query block: loops over key blocks kb <= qb. Also computes
// D_i = sum_d dO_i,d O_i,d for its rows and stores it for the dK/dV kernel.
__global__ void __launch_bounds__(128) flash_bwd_dq_k(bf16* __restrict__ dqkv,
                                                      const bf16* __restrict__ dout,
                                                      const bf16* __restrict__ qkv,
                                                      const bf16* __restrict__ outp,
                                                      const float* __restrict__ lse,
                                                      float* __restrict__ Dg, int Tn, int C,
                                                      int NH, float scale, float scale_log2) {
    __shared__ __align__(128) bf16 sQ[BLK * HSZ];
    __shared__ __align__(128) bf16 sdO[BLK * HSZ];
    __shared__ __align__(128) bf16 sK[2][BLK * HSZ];
    __shared__ __align__(128) bf16 sV[2][BLK * HSZ];
    const int qb = gridDim.x - 1 - blockIdx.x;
    const int b = blockIdx.y / NH, h = blockIdx.y % NH;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t pitch = 3 * (size_t)C;
    const bf16* Qg = qkv + (size_t)b * Tn * pitch + (size_t)h * HSZ;
    const bf16* Kg = Qg + C;
    const bf16* Vg = Qg + 2 * C;
    const bf16* dOg = dout + (size_t)b * Tn * C + (size_t)h * HSZ;
    load_tile(sQ, Qg, qb * BLK, Tn, pitch);
    load_tile(sdO, dOg, qb * BLK, Tn, (size_t)C);
    load_tile(sK[0], Kg, 0, Tn, pitch);
    load_tile(sV[0], Vg, 0, Tn, pitch);
    cp_commit();
    const size_t row_base = ((size_t)b * NH + h) * Tn;
    // D for the block's 64 rows: two threads per row, 32 elements each; warp w
    // computes exactly its own 16 rows, so the values are exchanged by shuffles
    float dacc = 0.f;
    {
        const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
        const int q = qb * BLK + r;
        if (q < Tn) {
            const bf16* o = outp + ((size_t)b * Tn + q) * C + (size_t)h * HSZ + half * 32;
            const bf16* g = dout + ((size_t)b * Tn + q) * C + (size_t)h * HSZ + half * 32;
#pragma unroll
            for (int v = 0; v < 4; v++) {
                Vec16<bf16> ov = ld16(o + 8 * v), gv = ld16(g + 8 * v);
#pragma unroll
                for (int k = 0; k < 8; k++) dacc += to_f(ov.v[k]) * to_f(gv.v[k]);
            }
        }
        dacc += __shfl_xor_sync(0xffffffffu, dacc, 1);
        if (half == 0 && q < Tn) Dg[row_base + q] = dacc;
    }
    float lse2[2], Dr[2];
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int q = qb * BLK + warp * 16 + (lane >> 2) + 8 * r;
        lse2[r] = q < Tn ? lse[row_base + q] * LOG2E_F : 0.f;
        Dr[r] = __shfl_sync(0xffffffffu, dacc, 2 * ((lane >> 2) + 8 * r));
    }
    uint32_t qf[4][4], df[4][4];
    float dq[8][4];
    zero_acc(dq);
    const int nkb = qb + 1;
    for (int kb = 0; kb < nkb; kb++) {
        if (kb + 1 < nkb) {
            load_tile(sK[(kb + 1) & 1], Kg, (kb + 1) * BLK, Tn, pitch);
            load_tile(sV[(kb + 1) & 1], Vg, (kb + 1) * BLK, Tn, pitch);
            cp_commit();
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        if (kb == 0) {
            load_a_frags(qf, sQ, warp * 16);
            load_a_frags(df, sdO, warp * 16);
        }
        float s[8][4], dp[8][4];
        zero_acc(s);
        zero_acc(dp);
        mma_abt(s, qf, sK[kb & 1]);
        mma_abt(dp, df, sV[kb & 1]);
        const int qr = warp * 16 + (lane >> 2);
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int r = e >> 1;
                float p = exp2f(s[nt][e] * scale_log2 - lse2[r]);
                if (kb == qb) {
                    const int key = nt * 8 + 2 * (lane & 3) + (e & 1);
                    if (key > qr + 8 * r) p = 0.f;
                }
                s[nt][e] = p * (dp[nt][e] - Dr[r]);  // dS
            }
        }
        mma_pv(dq, s, sK[kb & 1]);
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int q = qb * BLK + warp * 16 + (lane >> 2) + 8 * r;
        if (q < Tn) {
            bf16* dst = dqkv + ((size_t)b * Tn + q) * pitch + (size_t)h * HSZ;
#pragma unroll
            for (int nt = 0; nt < 8; nt++) {
                const int d = nt * 8 + 2 * (lane & 3);
                *reinterpret_cast<uint32_t*>(dst + d) =
                    pack_bf16(dq[nt][2 * r] * scale, dq[nt][2 * r + 1] * scale);
            }
        }
    }
}

// dK, dV for one key block: loops over query blocks qb >= kb
__global__ void __launch_bounds__(128) flash_bwd_dkv_k(bf16* __restrict__ dqkv,
                                                       const bf16* __restrict__ dout,
                                                       const bf16* __restrict__ qkv,
                                                       const float* __restrict__ lse,
                                                       const float* __restrict__ Dg, int Tn,
                                                       int C, int NH, float scale,
                                                       float scale_log2) {
    __shared__ __align__(128) bf16 sK[BLK * HSZ];
    __shared__ __align__(128) bf16 sV[BLK * HSZ];
    __shared__ __align__(128) bf16 sQ[2][BLK * HSZ];
    __shared__ __align__(128) bf16 sdO[2][BLK * HSZ];
    const int kb = blockIdx.x;  // smallest key block has the most query blocks: first
    const int b = blockIdx.y / NH, h = blockIdx.y % NH;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t pitch = 3 * (size_t)C;
    const bf16* Qg = qkv + (size_t)b * Tn * pitch + (size_t)h * HSZ;
    const bf16* Kg = Qg + C;
    const bf16* Vg = Qg + 2 * C;
    const bf16* dOg = dout + (size_t)b * Tn * C + (size_t)h * HSZ;
    const int nqb = (Tn + BLK - 1) / BLK;
    load_tile(sK, Kg, kb * BLK, Tn, pitch);
    load_tile(sV, Vg, kb * BLK, Tn, pitch);
    load_tile(sQ[0], Qg, kb * BLK, Tn, pitch);
    load_tile(sdO[0], dOg, kb * BLK, Tn, (size_t)C);
    cp_commit();
    const size_t row_base = ((size_t)b * NH + h) * Tn;
    uint32_t kf[4][4], vf[4][4];
    float dk[8][4], dv[8][4];
    zero_acc(dk);
    zero_acc(dv);
    const int kr = warp * 16 + (lane >> 2);  // key row within the block (and +8)
    for (int qb = kb; qb < nqb; qb++) {
        const int it = qb - kb;
        if (qb + 1 < nqb) {
            load_tile(sQ[(it + 1) & 1], Qg, (qb + 1) * BLK, Tn, pitch);
            load_tile(sdO[(it + 1) & 1], dOg, (qb + 1) * BLK, Tn, (size_t)C);
            cp_commit();
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();
        if (it == 0) {
            load_a_frags(kf, sK, warp * 16);
            load_a_frags(vf, sV, warp * 16);
        }
        float st[8][4], dpt[8][4];
        zero_acc(st);
        zero_acc(dpt);
        mma_abt(st, kf, sQ[it & 1]);    // S^T = K Q^T   (rows keys, cols queries)
        mma_abt(dpt, vf, sdO[it & 1]);  // dP^T = V dO^T
#pragma unroll
        for (int nt = 0; nt < 8; nt++) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int qi = qb * BLK + nt * 8 + 2 * (lane & 3) + (e & 1);
                const int key = kb * BLK + kr + ((e >> 1) << 3);
                float p = 0.f, dd = 0.f;
                if (qi < Tn && key <= qi) {
                    p = exp2f(st[nt][e] * scale_log2 - lse[row_base + qi] * LOG2E_F);
                    dd = Dg[row_base + qi];
                }
                st[nt][e] = p;                       // P^T
                dpt[nt][e] = p * (dpt[nt][e] - dd);  // dS^T
            }
        }
        mma_pv(dv, st, sdO[it & 1]);  // dV += P^T dO
        mma_pv(dk, dpt, sQ[it & 1]);  // dK += dS^T Q
        __syncthreads();
    }
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int key = kb * BLK + kr + 8 * r;
        if (key < Tn) {
            bf16* dkp = dqkv + ((size_t)b * Tn + key) * pitch + C + (size_t)h * HSZ;
            bf16* dvp = dkp + C;
#pragma unroll
            for (int nt = 0; nt < 8; nt++) {
                const int d = nt * 8 + 2 * (lane & 3);
                *reinterpret_cast<uint32_t*>(dkp + d) =
                    pack_bf16(dk[nt][2 * r] * scale, dk[nt][2 * r + 1] * scale);
                *reinterpret_cast<uint32_t*>(dvp + d) = pack_bf16(dv[nt][2 * r], dv[nt][2 * r + 1]);
            }
        }
    }
}

}  // namespace fa

// ================================================================== launchers
template <typename T>
static void simt_forward(void* out, float* lse, const void* qkv, int B, int Tn, int C, int NH,
                         cudaStream_t s) {
    const int HS = C / NH;
    const int n = B * NH * Tn;
    const int block = 128, grid = (n + block - 1) / block;
    switch (HS) {
        case 16: attn_fwd_simt_k<T, 16><<<grid, block, 0, s>>>((T*)out, lse, (const T*)qkv, B, Tn, C, NH); break;
        case 32: attn_fwd_simt_k<T, 32><<<grid, block, 0, s>>>((T*)out, lse, (const T*)qkv, B, Tn, C, NH); break;
        case 64: attn_fwd_simt_k<T, 64><<<grid, block, 0, s>>>((T*)out, lse, (const T*)qkv, B, Tn, C, NH); break;
        default: attn_fwd_simt_k<T, 128><<<grid, block, 0, s>>>((T*)out, lse, (const T*)qkv, B, Tn, C, NH); break;
    }
}

template <typename T>
static void simt_backward(void* dqkv, const void* dout, const void* qkv, const float* lse,
                          const float* D, int B, int Tn, int C, int NH, cudaStream_t s) {
    const int HS = C / NH;
    const int n = B * NH * Tn;
    const int block = 128, grid = (n + block - 1) / block;
#define ATTB(HSV)                                                                               \
    attn_bwd_dq_simt_k<T, HSV><<<grid, block, 0, s>>>((T*)dqkv, (const T*)dout, (const T*)qkv, \
                                                      lse, D, B, Tn, C, NH);                    \
    attn_bwd_dkv_simt_k<T, HSV><<<grid, block, 0, s>>>((T*)dqkv, (const T*)dout,               \
                                                       (const T*)qkv, lse, D, B, Tn, C, NH)
    switch (HS) {
        case 16: ATTB(16); break;
        case 32: ATTB(32); break;
        case 64: ATTB(64); break;
        default: ATTB(128); break;
    }
#undef ATTB
}

int launch_attention_forward(DType dt, int tensor_cores, void* out, float* lse, const void* qkv,
                             int B, int T, int C, int NH, cudaStream_t s, unsigned int* err) {
    const int HS = C / NH;
    if (dt == DT_F16 && tensor_cores && HS == 64) {
        // tcgen05 kernel (fp16 operands); the SIMT kernel for operands TMA cannot address
        const int rc = launch_flash_forward_tc(dt, out, lse, qkv, B, T, C, NH, s, err);
        if (rc != GPT2_ERR_ALIGN) return rc;
    }
    if (dt == DT_BF16 && tensor_cores && HS == 64) {
        // tcgen05 kernel; the m16n8k16 kernel remains for operands TMA cannot address
        const int rc = launch_flash_forward_tc(dt, out, lse, qkv, B, T, C, NH, s, err);
        if (rc != GPT2_ERR_ALIGN) return rc;
        note_launch(1);
        dim3 grid((T + fa::BLK - 1) / fa::BLK, B * NH);
        const float scale_log2 = LOG2E_F / sqrtf((float)HS);
        fa::flash_fwd_k<<<grid, 128, 0, s>>>((bf16*)out, lse, (const bf16*)qkv, T, C, NH, scale_log2);
        return GPT2_OK;
    }
    note_launch(1);
    if (dt == DT_BF16) simt_forward<bf16>(out, lse, qkv, B, T, C, NH, s);
    else if (dt == DT_F16) simt_forward<f16>(out, lse, qkv, B, T, C, NH, s);
    else simt_forward<float>(out, lse, qkv, B, T, C, NH, s);
    return GPT2_OK;
}

int launch_attention_backward(DType dt, int tensor_cores, void* dqkv, const void* dout,
                              const void* qkv, const void* out, const float* lse, float* D, int B,
                              int T, int C, int NH, cudaStream_t s, unsigned int* err) {
    const int HS = C / NH;
    const int n = B * NH * T;
    if (dt == DT_F16 && tensor_cores && HS == 64) {
        // tcgen05 kernels (fp16 operands); the SIMT kernels for operands TMA cannot address
        const int rc = launch_flash_backward_tc(dt, dqkv, dout, qkv, out, lse, D, B, T, C, NH, s, err);
        if (rc != GPT2_ERR_ALIGN) return rc;
    }
    if (dt == DT_BF16 && tensor_cores && HS == 64) {
        // tcgen05 kernels; the m16n8k16 kernels remain for operands TMA cannot address
        const int rc = launch_flash_backward_tc(dt, dqkv, dout, qkv, out, lse, D, B, T, C, NH, s, err);
        if (rc != GPT2_ERR_ALIGN) return rc;
        note_launch(2);
        dim3 grid((T + fa::BLK - 1) / fa::BLK, B * NH);
        const float scale = 1.f / sqrtf((float)HS), scale_log2 = LOG2E_F * scale;
        fa::flash_bwd_dq_k<<<grid, 128, 0, s>>>((bf16*)dqkv, (const bf16*)dout, (const bf16*)qkv,
                                                (const bf16*)out, lse, D, T, C, NH, scale,
                                                scale_log2);
        fa::flash_bwd_dkv_k<<<grid, 128, 0, s>>>((bf16*)dqkv, (const bf16*)dout, (const bf16*)qkv,
                                                 lse, D, T, C, NH, scale, scale_log2);
        return GPT2_OK;
    }
    note_launch(3);
    if (dt == DT_BF16)
        attn_rowdot_k<bf16><<<(n + 255) / 256, 256, 0, s>>>(D, (const bf16*)dout, (const bf16*)out,
                                                            B, T, C, NH, HS);
    else if (dt == DT_F16)
        attn_rowdot_k<f16><<<(n + 255) / 256, 256, 0, s>>>(D, (const f16*)dout, (const f16*)out,
                                                           B, T, C, NH, HS);
    else
        attn_rowdot_k<float><<<(n + 255) / 256, 256, 0, s>>>(D, (const float*)dout,
                                                             (const float*)out, B, T, C, NH, HS);
    if (dt == DT_BF16) simt_backward<bf16>(dqkv, dout, qkv, lse, D, B, T, C, NH, s);
    else if (dt == DT_F16) simt_backward<f16>(dqkv, dout, qkv, lse, D, B, T, C, NH, s);
    else simt_backward<float>(dqkv, dout, qkv, lse, D, B, T, C, NH, s);
    return GPT2_OK;
}

}  // namespace gk
