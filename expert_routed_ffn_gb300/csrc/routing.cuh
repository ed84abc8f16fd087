// The routing rule of one token (K1), shared by the tensor-core router and
// the CUDA-core router: scores, selection-only bias, top-k with lower-index
// tie-break, weights from the unbiased scores, route_norm, route_scale
// (Arcee AFMoE issue, "Routing detail"; HF AFMoE docs, "expert routing").
#pragma once

#include "common.cuh"

namespace moe {

// Selection key of a candidate: a larger key is a larger biased score c, and among
// equal c the lower expert index e.  High word: c as an order-preserving integer (c is
// never NaN here; -0 is taken as +0, they compare equal); low word: 0xFFFF - e.  The
// key 0 sorts below every candidate, even c = -inf.
__device__ __forceinline__ unsigned long long sel_key(float c, int e) {
    uint32_t u = __float_as_uint(c == 0.f ? 0.f : c);
    u ^= (u >> 31) ? 0xFFFFFFFFu : 0x80000000u;
    return ((unsigned long long)u << 32) | (uint32_t)(0xFFFF - e);
}
__device__ __forceinline__ void cas_desc(unsigned long long &a, unsigned long long &b) {
    const unsigned long long hi = a > b ? a : b, lo = a > b ? b : a;
    a = hi;
    b = lo;
}
// The 8 keys of this lane in descending order (a bitonic sorting network).
__device__ __forceinline__ void sort8_desc(unsigned long long (&k)[8]) {
#pragma unroll
    for (int size = 2; size <= 8; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    if ((i & size) == 0)
                        cas_desc(k[i], k[j]);
                    else
                        cas_desc(k[j], k[i]);
                }
            }
}

// The routing rule for one token, by a group of LPT consecutive lanes: lane
// `sub` of the group holds the logits of 8 experts in lg[0..7] (E <= 8*LPT):
// experts sub, sub+LPT, ... (strided) or experts 8*sub .. 8*sub+7 (CONTIG).
// s = sigmoid(l) (or softmax over e); k times, the largest s + bias among the
// experts not chosen yet (equal values: lower expert index) is chosen; weights
// from the unbiased s, renormalised when route_norm is set, then times
// route_scale.  Every lane of the warp must call it (shuffles); only groups
// with `valid` write slots (lane sub writes slots r = sub mod LPT) and count
// the chosen experts in hist (shared memory) when it is given.
template <int LPT, bool CONTIG = false>
__device__ __forceinline__ void route_token_group(const float (&lg)[8], int sub, bool valid, int t, int E,
                                                  int k, const float *bias, int score_func, int route_norm,
                                                  float route_scale, int32_t *topk_idx, float *topk_w,
                                                  int *hist) {
    auto expert_of = [&](int j) { return CONTIG ? 8 * sub + j : sub + LPT * j; };
    float s[8], c[8];
    if (score_func == 1) {
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (expert_of(j) < E) m = fmaxf(m, lg[j]);
#pragma unroll
        for (int o = LPT / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o, LPT));
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            s[j] = (expert_of(j) < E) ? expf(lg[j] - m) : 0.f;
            z += s[j];
        }
#pragma unroll
        for (int o = LPT / 2; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o, LPT);
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j] = s[j] / z;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j] = 1.0f / (1.0f + expf(-lg[j]));
    }
    // Each lane sorts its candidates' selection keys once; a round then takes the
    // largest head over the group (log2(LPT) shuffle levels, no scan of the candidates)
    // and the lane that held it drops its head.
    unsigned long long key[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = expert_of(j);
        if (e < E) {
            float cj = s[j] + (bias ? __ldg(bias + e) : 0.f);
            cj = (cj != cj) ? -INFINITY : cj;  // NaN never wins
            key[j] = sel_key(cj, e);
        } else {
            key[j] = 0ull;
        }
    }
    sort8_desc(key);
    // Slot r is kept by lane r mod LPT of the group (entry r / LPT of its
    // own[] arrays), so the k rounds compile to one loop body: the routing
    // kernels run once per forward with a cold instruction cache.
    constexpr int kOwn = (16 + LPT - 1) / LPT;
    float own_s[kOwn];
    int own_e[kOwn];
#pragma unroll
    for (int q = 0; q < kOwn; ++q) {
        own_s[q] = 0.f;
        own_e[q] = 0;
    }
    float wsum = 0.f;
#pragma unroll 1
    for (int r = 0; r < k; ++r) {
        unsigned long long best = key[0];
#pragma unroll
        for (int o = LPT / 2; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o, LPT);
            best = other > best ? other : best;
        }
        if (key[0] == best) {  // this lane's head was chosen (keys are unique)
#pragma unroll
            for (int q = 0; q < 7; ++q) key[q] = key[q + 1];
            key[7] = 0ull;
        }
        const int be = 0xFFFF - (int)(uint32_t)(best & 0xFFFFull);
        const int owner = CONTIG ? be >> 3 : be & (LPT - 1), jj = CONTIG ? be & 7 : be / LPT;
        float sv = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (q == jj) sv = s[q];
        sv = __shfl_sync(0xffffffffu, sv, owner, LPT);
        wsum += sv;
        if ((r & (LPT - 1)) == sub) {
            const int qr = r / LPT;
#pragma unroll
            for (int q = 0; q < kOwn; ++q)
                if (q == qr) {
                    own_s[q] = sv;
                    own_e[q] = be;
                }
        }
    }
    if (valid) {
#pragma unroll
        for (int q = 0; q < kOwn; ++q) {
            const int r = sub + LPT * q;
            if (r < k) {
                float w = own_s[q];
                if (route_norm) w = w / wsum;
                w = w * route_scale;
                topk_idx[(size_t)t * k + r] = own_e[q];
                topk_w[(size_t)t * k + r] = w;
                if (hist != nullptr) atomicAdd(&hist[own_e[q]], 1);
            }
        }
    }
}

}  // namespace moe
