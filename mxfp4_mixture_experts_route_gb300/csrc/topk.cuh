// Sigmoid top-k of one token by one warp (shared by the top-k kernel and the
// fused top-k + sort + gather kernel).
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

// The lane's slots of the bias (lane l holds experts l, l + 32, ...).
template <int MAXE>
__device__ __forceinline__ void load_bias(const float* __restrict__ bias, int E, int lane, float (&b)[MAXE]) {
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
        const int e = lane + 32 * i;
        b[i] = e < E ? bias[e] : 0.f;
    }
}

// A token's logits (the router's output, read through L2): lane l gets
// experts l, l + 32, ... (independent loads, all in flight together).
template <int MAXE>
__device__ __forceinline__ void topk_load(const float* Lrow, int E, int lane, float (&z)[MAXE]) {
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
        const int e = lane + 32 * i;
        z[i] = e < E ? ld_dep(Lrow + e) : 0.f;
    }
}

// The top k of one token from its logits z (topk_load) and the bias b
// (load_bias), by one warp; s_sh is the warp's scratch of 32 * MAXE floats in
// shared memory.
//   1. each expert's entry v = key << 32 | ~id orders by score, then by lower
//      id; every lane sorts its MAXE entries (a bitonic network in registers,
//      independent of the other lanes)
//   2. k rounds: the largest key among the lanes' heads (one redux), the
//      lowest id among the heads that hold it (a second redux; a lane's other
//      entries of that key have higher ids than its head); the owning lane
//      drops its head, lane r keeps round r's winner
//   3. lane j < k: the rank of its id among the k (ascending id order), its s
//      from s_sh and the sum of the picks' s (a butterfly over the lanes, the
//      same in all)
// On return lane j < k holds one pick: its id, its weight and its rank in
// ascending id order (the caller writes it to slot rank).
template <int MAXE>
__device__ __forceinline__ void topk_select(const float (&z)[MAXE], const float (&b)[MAXE], int E, int k, int lane,
                                            float* s_sh, int& id_out, float& w_out, int& rank_out) {
    uint64_t v[MAXE];
#pragma unroll
    for (int i = 0; i < MAXE; ++i) {
        const int e = lane + 32 * i;
        const float s = __fdividef(1.0f, 1.0f + __expf(-z[i]));   // a few ulp; the sets need score gaps far larger
        s_sh[e] = s;
        const uint32_t key = e < E ? sel_key(s + b[i]) : 0u;
        v[i] = (uint64_t)key << 32 | (uint64_t)(~(uint32_t)e);
    }
    // 1: descending
#pragma unroll
    for (int kk = 2; kk <= MAXE; kk <<= 1) {
#pragma unroll
        for (int j = kk >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < MAXE; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    const uint64_t x0 = v[i], x1 = v[l];
                    const bool sw = (i & kk) == 0 ? x1 > x0 : x0 > x1;
                    v[i] = sw ? x1 : x0;
                    v[l] = sw ? x0 : x1;
                }
            }
        }
    }
    // 2
    int my_id = 0x7fffffff;
    for (int r = 0; r < k; ++r) {
        const uint32_t hk = (uint32_t)(v[0] >> 32);
        const uint32_t m = __reduce_max_sync(0xffffffffu, hk);
        const uint32_t win = __reduce_min_sync(0xffffffffu, hk == m ? ~(uint32_t)v[0] : 0xffffffffu);
        const bool own = (int)(win & 31u) == lane;
#pragma unroll
        for (int i = 0; i + 1 < MAXE; ++i) v[i] = own ? v[i + 1] : v[i];
        v[MAXE - 1] = own ? 0ull : v[MAXE - 1];
        my_id = lane == r ? (int)win : my_id;
    }
    // 3
    __syncwarp();
    int rank = 0;
    for (int j = 0; j < k; ++j) rank += __shfl_sync(0xffffffffu, my_id, j) < my_id ? 1 : 0;
    const float sv = lane < k ? s_sh[my_id] : 0.f;
    float tot = sv;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    id_out = my_id;
    w_out = sv / tot;
    rank_out = rank;
    __syncwarp();   // s_sh is written again by the warp's next token
}

}  // namespace moe
