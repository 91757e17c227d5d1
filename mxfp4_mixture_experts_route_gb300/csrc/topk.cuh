// Sigmoid top-k of one token by one warp (shared by the top-k kernel and the
// fused top-k + sort kernel).
//
// vllm.models.muse_spark.amd.mono.kernels.k3, route_token (sigmoid scores);
// k5, stage HA (top 8, ids and weights out).  s = sigmoid(L), sel = s + bias;
// the k largest sel win (ties -> lower expert id), reported in ascending id
// order with w_j = s_j / sum of the picks' s.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// 32-bit key ordered like the selection score: a larger score has a larger
// key.  NaN gets 1 (below every number); 0 marks a slot out of the race.
__device__ __forceinline__ uint32_t sel_key(float v) {
    if (v != v) return 1u;
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The lane's best slot: largest key, lowest slot on ties (a pairwise tree in
// which the left operand always holds the lower slots).
template <int MAXE>
__device__ __forceinline__ void lane_best(const uint32_t (&key)[MAXE], uint32_t& bk, int& bi) {
    uint32_t kk[MAXE];
    int ii[MAXE];
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
        kk[i] = key[i];
        ii[i] = i;
    }
#pragma unroll
    for (int st = 1; st < MAXE; st <<= 1) {
#pragma unroll
        for (int i = 0; i + st < MAXE; i += 2 * st) {
            const bool take = kk[i + st] > kk[i];
            kk[i] = take ? kk[i + st] : kk[i];
            ii[i] = take ? ii[i + st] : ii[i];
        }
    }
    bk = kk[0];
    bi = ii[0];
}

// The lane's slots of the bias (lane l holds experts l, l + 32, ...).
template <int MAXE>
__device__ __forceinline__ void load_bias(const float* __restrict__ bias, int E, int lane, float (&b)[MAXE]) {
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
        const int e = lane + 32 * i;
        b[i] = e < E ? bias[e] : 0.f;
    }
}

// Lane l holds experts l, l + 32, ... (E <= 32 * MAXE), b from load_bias.
// Each round takes the warp's largest key (one redux), the lowest expert id
// among the lanes that hold it (a second redux), and lets the owning lane
// retire it and find its next best.  Writes ids_out[0..k) in ascending id and
// w_out[0..k).
template <int MAXE>
__device__ __forceinline__ void topk_token(const float* Lrow, const float (&b)[MAXE], int E, int k,
                                           int lane, int32_t* ids_out, float* w_out) {
    float s[MAXE], z[MAXE];
    uint32_t key[MAXE];
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {           // independent loads, all in flight together
        const int e = lane + 32 * i;
        z[i] = e < E ? ld_dep(Lrow + e) : 0.f;   // the router's output
    }
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
        const int e = lane + 32 * i;
        s[i] = __fdividef(1.0f, 1.0f + __expf(-z[i]));   // a few ulp; the sets need score gaps far larger
        key[i] = e < E ? sel_key(s[i] + b[i]) : 0u;
    }
    uint32_t bk;
    int bi;
    lane_best(key, bk, bi);
    int my_id = 0x7fffffff;   // lane j < k keeps pick j
    float my_s = 0.f;
    for (int r = 0; r < k; ++r) {
        const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t win = __reduce_min_sync(0xffffffffu, bk == m ? (uint32_t)(lane + 32 * bi) : 0xffffffffu);
        const int owner = (int)(win & 31u);
        float sv = 0.f;
        if (lane == owner) {
            const int slot = (int)(win >> 5);
#pragma unroll
            for (int i = 0; i < MAXE; ++i) {
                if (i == slot) {
                    sv = s[i];
                    key[i] = 0u;
                }
            }
            lane_best(key, bk, bi);
        }
        sv = __shfl_sync(0xffffffffu, sv, owner);
        if (lane == r) {
            my_id = (int)win;
            my_s = sv;
        }
    }
    // ascending id order: rank of my pick among the k picks
    float tot = 0.f;
    int rank = 0;
    for (int j = 0; j < k; ++j) {
        const int oid = __shfl_sync(0xffffffffu, my_id, j);
        tot += __shfl_sync(0xffffffffu, my_s, j);
        rank += (oid < my_id) ? 1 : 0;
    }
    if (lane < k) {
        ids_out[rank] = my_id;
        w_out[rank] = my_s / tot;
    }
}

}  // namespace moe
