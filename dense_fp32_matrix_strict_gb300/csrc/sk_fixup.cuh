// sk_fixup.cuh — the stream-K tail's epilogue kernel: adds the partial sums
// the SGEMM kernel left in workspace slots for split tiles, in k order, and
// applies C = alpha * sum + beta * C.
#pragma once

#include "sgemm_kernel.cuh"

namespace sg {

// Most partial segments a stream-K tile can have; the host never schedules
// more (a range is at least ceil(k_tiles / 32) iterations long).
constexpr int kSkMaxParts = 64;

// The workspace slots holding the partial sums of stream-K tile u (tile
// dp_tiles + u), in increasing k order: the ranges of CTAs c_first,
// c_first + 1, ... that touch the tile, slot 2c for a range's first segment
// and 2c + 1 for a later one. Returns their number (0 if one range covered
// the tile whole, which that CTA then finished itself), or -1 past
// kSkMaxParts.
__device__ __forceinline__ int sk_parts(const GemmParams& p, long long u, int* parts) {
    const long long KT = p.k_tiles, G = p.sk_ctas, S = p.sk_iters;
    const long long x0 = u * KT, x1 = x0 + KT;
    // Largest c with start(c) <= x0: the range holding the tile's first k.
    long long c = ((x0 + 1) * G + S - 1) / S - 1;
    if (c < 0) c = 0;
    int n = 0;
    for (; c < G; ++c) {
        const long long s = sk_start(c, p), e = sk_start(c + 1, p);
        if (s >= x1) break;
        const long long a = s > x0 ? s : x0;
        const long long b = e < x1 ? e : x1;
        if (a >= b) continue;
        if (a == x0 && b == x1) return 0;
        if (n == kSkMaxParts) return -1;
        parts[n++] = static_cast<int>(2 * c + (a == s ? 0 : 1));
    }
    return n;
}

// `split` CTAs per stream-K tile u (tile dp_tiles + u), each taking one
// contiguous share of the tile's float4s, so the fixup fills the GPU even
// when few tiles are split. Each float4 is alpha * (the np partial slots
// added in k order) + beta * C, with the vector and scalar rules of the
// epilogue; the slot loads of one float4 are issued four at a time (L2
// reads, ld.global.cg) before they are added in order, so every thread keeps
// several in flight.
template <int BM, int BN>
__global__ void __launch_bounds__(256)
sk_fixup_kernel(const GemmParams p, int split) {
    const long long u = blockIdx.x / split;
    const int part = static_cast<int>(blockIdx.x % split);
    __shared__ int parts[kSkMaxParts];
    __shared__ int nparts;
    if (threadIdx.x == 0) {
        const int n = sk_parts(p, u, parts);
        if (n < 0) atomicOr(p.status, STATUS_SCHEDULE);
        nparts = n < 0 ? 0 : n;
    }
    __syncthreads();
    const int np = nparts;
    if (np == 0) return;

    int tm, tn;
    tile_coords(p.dp_tiles + static_cast<int>(u), p, tm, tn);
    const bool use_c = p.beta != 0.0f;
    constexpr int Q = BM * BN / 4;              // float4 per tile
    constexpr long long SLOT = BM * BN / 4;     // float4 per slot
    const int per = (Q + split - 1) / split;
    const int q1 = (part + 1) * per < Q ? (part + 1) * per : Q;
    const float4* __restrict__ ws = reinterpret_cast<const float4*>(p.ws);
#pragma unroll 1
    for (int q = part * per + static_cast<int>(threadIdx.x); q < q1; q += blockDim.x) {
        const int r = q / (BN / 4);
        const int c4 = (q - r * (BN / 4)) * 4;
        const int m = tm * BM + r;
        const int n = tn * BN + c4;
        if (m >= p.M || n >= p.N) continue;
        const float4* src = ws + q;
        SG_DCHECK(p, q < Q && parts[0] >= 0 && parts[np - 1] < 2 * p.sk_ctas);
        float4 sum = __ldcg(src + parts[0] * SLOT);
        int j = 1;
#pragma unroll 1
        for (; j + 4 <= np; j += 4) {
            const float4 v0 = __ldcg(src + parts[j] * SLOT);
            const float4 v1 = __ldcg(src + parts[j + 1] * SLOT);
            const float4 v2 = __ldcg(src + parts[j + 2] * SLOT);
            const float4 v3 = __ldcg(src + parts[j + 3] * SLOT);
            sum.x += v0.x; sum.y += v0.y; sum.z += v0.z; sum.w += v0.w;
            sum.x += v1.x; sum.y += v1.y; sum.z += v1.z; sum.w += v1.w;
            sum.x += v2.x; sum.y += v2.y; sum.z += v2.z; sum.w += v2.w;
            sum.x += v3.x; sum.y += v3.y; sum.z += v3.z; sum.w += v3.w;
        }
        for (; j < np; ++j) {
            const float4 v = __ldcg(src + parts[j] * SLOT);
            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
        }
        float* crow = p.C + (long long)m * p.ldc;
        float v[4] = {p.alpha * sum.x, p.alpha * sum.y, p.alpha * sum.z, p.alpha * sum.w};
        if (p.c_vec && n + 3 < p.N) {
            float4* cp = reinterpret_cast<float4*>(crow + n);
            if (use_c) {
                const float4 cv = *cp;
                v[0] = fmaf(p.beta, cv.x, v[0]);
                v[1] = fmaf(p.beta, cv.y, v[1]);
                v[2] = fmaf(p.beta, cv.z, v[2]);
                v[3] = fmaf(p.beta, cv.w, v[3]);
            }
            *cp = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            for (int e = 0; e < 4; ++e) {
                if (n + e < p.N) {
                    float out = v[e];
                    if (use_c) out = fmaf(p.beta, crow[n + e], out);
                    crow[n + e] = out;
                }
            }
        }
    }
}

}  // namespace sg
