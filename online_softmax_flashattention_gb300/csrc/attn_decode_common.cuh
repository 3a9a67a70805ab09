// Work split of the key-value cache path, shared by the CUDA-core and tensor-core decode kernels
// and the merge kernel (see attn_decode.cu for the plan these describe).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace attn {

struct DecodeParams {
    const void* q;
    void* o;
    float* lse;       // null, or [BH, Nq]
    float* part_o;    // [BH * Nq][P][D]
    float* part_lse;  // [BH * Nq][P]
    int Nq, Nk, BH;
    int groups;           // query groups per head
    int Tn;               // tiles per segment
    int causal;
    int explicit_splits;  // S >= 1: every segment in S shares; 0: balanced
    int tps;              // explicit: tiles per share
    int P;                // slot stride of the partials (S, or most pieces a segment can have)
    int C;                // CTAs in the grid
    int64_t G;            // balanced: segments * Tn
    float c;              // log2(e) / sqrt(D)
};

struct Piece {
    int bh, g0, ng;  // head, first query of the group, queries in the group
    int t0, t1;      // tiles [t0, t1) of the segment, already clipped to the visible keys
    int ke;          // the segment's visible keys end before ke
    int slot, nslots;
};

// Balanced mode: the CTA whose run holds global tile t.
__device__ __host__ inline int64_t owner_of(int64_t t, int64_t C, int64_t G) {
    return ((t + 1) * C - 1) / G;
}

// The k-th piece of CTA `cta` (tiles of ROWS keys); false once the CTA has no more.
template <int QG, int ROWS>
__device__ inline bool get_piece(const DecodeParams& p, int cta, int k, Piece& pc) {
    int64_t seg;
    int t0, t1;
    if (p.explicit_splits > 0) {
        const int64_t idx = static_cast<int64_t>(cta) + static_cast<int64_t>(k) * p.C;
        const int64_t nseg = static_cast<int64_t>(p.BH) * p.groups;
        if (idx >= nseg * p.explicit_splits) return false;
        seg = idx / p.explicit_splits;
        const int share = static_cast<int>(idx % p.explicit_splits);
        t0 = min(p.Tn, share * p.tps);
        t1 = min(p.Tn, t0 + p.tps);
        pc.slot = share;
        pc.nslots = p.explicit_splits;
    } else {
        const int64_t A = static_cast<int64_t>(cta) * p.G / p.C;
        const int64_t Bend = (static_cast<int64_t>(cta) + 1) * p.G / p.C;
        if (A >= Bend) return false;
        seg = A / p.Tn + k;
        const int64_t s0 = seg * p.Tn;
        if (s0 >= Bend) return false;
        const int64_t a = max(A, s0), b = min(Bend, s0 + p.Tn);
        t0 = static_cast<int>(a - s0);
        t1 = static_cast<int>(b - s0);
        const int64_t first = owner_of(s0, p.C, p.G), last = owner_of(s0 + p.Tn - 1, p.C, p.G);
        pc.slot = static_cast<int>(cta - first);
        pc.nslots = static_cast<int>(last - first + 1);
    }
    pc.bh = static_cast<int>(seg / p.groups);
    pc.g0 = static_cast<int>(seg % p.groups) * QG;
    pc.ng = min(QG, p.Nq - pc.g0);
    pc.ke = p.causal ? min(p.Nk, p.Nk - p.Nq + pc.g0 + pc.ng) : p.Nk;
    const int tv = (pc.ke + ROWS - 1) / ROWS;  // tiles holding a visible key
    pc.t0 = min(t0, tv);
    pc.t1 = min(t1, tv);
    return true;
}

// Tensor-core decode (attn_decode_tc.cu): launches its main kernel over prm.C CTAs (query groups of
// 128 rows; key tiles of 128 keys at d = 64, 64 at d = 128) with tensor maps of q ([BH][Nq][d],
// boxes of 128 rows x 64 values) and k, v ([BH][Nk][d], boxes of a key tile's rows x 64 values);
// bf16 or fp16.
int launch_decode_tc_main(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const DecodeParams& prm,
                          bool bf16, int d, cudaStream_t stream);

}  // namespace attn
