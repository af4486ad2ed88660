// sk_fixup.cuh — the stream-K tail's epilogue kernel: adds the partial sums
// the SGEMM kernel left in workspace slots for split tiles, in k order, and
// applies C = alpha * sum + beta * C.
#pragma once

#include "sgemm_kernel.cuh"

namespace sg {

// Most partial segments a stream-K tile can have; the host never schedules
// more (a range is at least ceil(k_tiles / kMaxParts) iterations long).
constexpr int kSkMaxParts = 64;

// `split` CTAs per stream-K tile u (tile dp_tiles + u), each taking one
// contiguous share of the tile's float4s, so the fixup fills the GPU even
// when few tiles are split. If a single CTA's range covered the whole tile,
// that CTA already wrote C and these blocks return. Otherwise the
// contributing ranges are those of CTAs c_first, c_first+1, ... (in
// increasing k order); their partial sums are added in that order and the
// epilogue C = alpha * sum + beta * C is applied.
template <int BM, int BN>
__global__ void __launch_bounds__(256)
sk_fixup_kernel(const GemmParams p, int split) {
    const long long KT = p.k_tiles;
    const long long G = p.sk_ctas;
    const long long S = p.sk_iters;
    const long long u = blockIdx.x / split;
    const int part = static_cast<int>(blockIdx.x % split);
    const long long x0 = u * KT, x1 = x0 + KT;
    __shared__ int parts[kSkMaxParts];
    __shared__ int nparts;
    if (threadIdx.x == 0) {
        // Largest c with start(c) <= x0: the range holding the tile's first k.
        long long c = ((x0 + 1) * G + S - 1) / S - 1;
        if (c < 0) c = 0;
        int n = 0;
        bool whole = false;
        for (; c < G; ++c) {
            const long long s = sk_start(c, p), e = sk_start(c + 1, p);
            if (s >= x1) break;
            const long long a = s > x0 ? s : x0;
            const long long b = e < x1 ? e : x1;
            if (a >= b) continue;
            if (a == x0 && b == x1) { whole = true; break; }
            if (n < kSkMaxParts) parts[n] = static_cast<int>(2 * c + (a == s ? 0 : 1));
            ++n;
        }
        nparts = whole ? 0 : n;
        if (n > kSkMaxParts) {
            atomicOr(p.status, STATUS_SCHEDULE);
            nparts = 0;
        }
    }
    __syncthreads();
    const int np = nparts;
    if (np == 0) return;

    int tm, tn;
    tile_coords(p.dp_tiles + static_cast<int>(u), p, tm, tn);
    const bool use_c = p.beta != 0.0f;
    constexpr int Q = BM * BN / 4;   // float4 per tile
    const int per = (Q + split - 1) / split;
    const int q1 = (part + 1) * per < Q ? (part + 1) * per : Q;
    for (int q = part * per + threadIdx.x; q < q1; q += blockDim.x) {
        const int r = q / (BN / 4);
        const int c4 = (q - r * (BN / 4)) * 4;
        const int m = tm * BM + r;
        const int n = tn * BN + c4;
        if (m >= p.M || n >= p.N) continue;
        float4 sum = __ldcg(reinterpret_cast<const float4*>(p.ws + static_cast<long long>(parts[0]) * (BM * BN)) + q);
        for (int j = 1; j < np; ++j) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p.ws + static_cast<long long>(parts[j]) * (BM * BN)) + q);
            sum.x += v.x;
            sum.y += v.y;
            sum.z += v.z;
            sum.w += v.w;
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
