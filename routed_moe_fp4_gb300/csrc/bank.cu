// Expert residency bank: S device slots that hold routed experts whose master copy lives in
// page-locked host memory, refilled route-aware on the device.
//
// The pages keep the most used routed experts of each layer resident on the GPU, ranked by
// usage, and refill that cache in place ("DeepSeek V4 Flash support -- CUDA/VRAM expert
// tiering", summary item 1; "the CUDA tier wired into the DeepSeek V4 engine", engine tier);
// for a batched prefill they route on the device and refill a transient per-layer bank in
// slot-sized groups, one group's uploads overlapped with its neighbour's compute (same page,
// prefill MoE). Here the host link is NVLink-C2C and the GPU reads the mapped host copy
// itself, so the plan, the refill and the GEMM rounds are all stream-ordered device work: the
// host never learns which experts a forward touched.
//
// One forward over the bank (api.cu runs it):
//   router, permute -> bank_plan -> x terms -> round 0 .. R-1: [bank_refill on the copy stream]
//   -> gate/up + down over that round's tiles -> combine.
// bank_plan decides, from cnt, which slot every touched expert computes from, which experts are
// copied in which round, and writes each round's n-tile records with the slot in the group
// field, so the FP4 GEMM runs over the bank unchanged.
//
// Policy (the pages give no more than the above; these are readings):
//  - cache forward (the host picks it when T*k or E, whichever is smaller, fits in S): resident
//    touched experts compute in place in round 0 with the shared expert; the others, in
//    increasing expert order, take the slots that are empty or hold an untouched expert,
//    smallest first by (occupied, usage of the expert, forward that last used the slot, slot);
//    they are copied and computed in round 1, while round 0 computes.
//  - transient forward otherwise: with G = S/2 the touched experts in increasing order form
//    groups of G; group r is round r and uses slots (r mod 2)*G + i, so round r+1's copies go to
//    the half that round r does not read. An expert already in its slot (rounds 0 and 1) is not
//    copied; one that moves leaves its old slot empty.
#include "block_scan.cuh"
#include "colimoe_internal.cuh"

namespace colimoe {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kErrBankSlots = 21;   // device error: a cache forward found no free slot
constexpr int kErrBankCopy = 22;    // device error: a refill entry out of range

struct PlanArgs {
    BankDev b;
    const int32_t *cnt, *off;
    int cache, G, R, ntile;
    int *err;
};

// Slot a is a better victim than slot b (cache forward): empty first, then the least used
// expert, then the slot used longest ago, then the lower slot.
__device__ __forceinline__ bool victim_less(int a, int b, const int *occ, const uint32_t *use, const int *last) {
    if ((occ[a] >= 0) != (occ[b] >= 0)) return occ[a] < 0;
    if (occ[a] >= 0) {
        if (use[a] != use[b]) return use[a] < use[b];
        if (last[a] != last[b]) return last[a] < last[b];
    }
    return a < b;
}

// One block of 1024 threads; thread e handles routed expert e (E <= 1024), thread s slot s.
__global__ void __launch_bounds__(kPlanThreads) bank_plan(PlanArgs a) {
    pdl_begin();
    __shared__ int scan_smem[33];
    __shared__ int s_occ[1024];          // slot -> expert before the forward
    __shared__ uint32_t s_use[1024];     // cache: usage of the slot's expert; transient: new occupant
    __shared__ int s_last[1024];         // cache: last use of the slot; transient: expert by rank
    __shared__ int s_aux[1024];          // cache: candidate flag, then victim by rank
    __shared__ int s_order[1024];        // order index -> expert
    __shared__ int s_oslot[1024];        // order index -> slot
    __shared__ int s_oround[1024];       // order index -> round
    __shared__ int s_rs[1024], s_ls[1024], s_cs[1024];   // per round: scan values of its first member
    __shared__ int s_step, s_sh_small, s_sh_large;
    const BankDev &b = a.b;
    const int tid = threadIdx.x, E = b.E, S = b.S;
    if (tid == 0) {
        s_step = (int)(b.stats[0] + 1);
        s_sh_small = 0;
        s_sh_large = 0;
    }
    for (int r = tid; r < a.R; r += kPlanThreads) {   // rounds without members stay empty
        b.counts[2 * r] = 0;
        b.counts[2 * r + 1] = 0;
        b.ncopy[r] = 0;
    }
    const int c = tid < E ? a.cnt[tid] : 0;
    const bool touched = c > 0;
    if (tid < S) s_occ[tid] = b.expert_in[tid];
    const int pre_slot = tid < E ? b.slot_of[tid] : -1;
    if (touched) b.usage[tid] += 1;
    int U;
    const int rank = block_exclusive_scan(touched ? 1 : 0, scan_smem, &U);   // syncs
    const int step = s_step;
    int o = -1, round = -1, slot = -1, copy = 0, H = 0;

    if (a.cache) {
        const bool hit = touched && pre_slot >= 0, miss = touched && pre_slot < 0;
        const int hrank = block_exclusive_scan(hit ? 1 : 0, scan_smem, &H);
        int M;
        const int mrank = block_exclusive_scan(miss ? 1 : 0, scan_smem, &M);
        if (tid < S) {
            const int occ = s_occ[tid];
            const bool cand = occ < 0 || a.cnt[occ] == 0;
            s_use[tid] = cand && occ >= 0 ? b.usage[occ] : 0u;   // untouched: unchanged by this forward
            s_last[tid] = b.last_use[tid];
            s_aux[tid] = cand ? 1 : 0;
        }
        __syncthreads();
        int vr = -1;
        if (tid < S && s_aux[tid]) {
            vr = 0;
            for (int s2 = 0; s2 < S; ++s2)
                if (s_aux[s2] && victim_less(s2, tid, s_occ, s_use, s_last)) ++vr;
        }
        int ncand;
        block_exclusive_scan(vr >= 0 ? 1 : 0, scan_smem, &ncand);   // syncs: s_aux reads are done
        if (vr >= 0) s_aux[vr] = tid;                               // victim by rank
        __syncthreads();
        if (hit) {
            o = hrank;
            round = 0;
            slot = pre_slot;
        } else if (miss) {
            o = H + mrank;
            round = 1;
            copy = 1;
            if (mrank < ncand) {
                slot = s_aux[mrank];
            } else {   // cannot happen when T*k or E fits in S
                slot = 0;
                copy = 0;
                atomicCAS(a.err, 0, kErrBankSlots);
            }
        }
        if (miss && copy && s_occ[slot] >= 0) b.slot_of[s_occ[slot]] = -1;   // evict (untouched)
        __syncthreads();
        if (miss && copy) {
            b.slot_of[tid] = slot;
            b.expert_in[slot] = tid;
        }
        if (touched) b.last_use[slot] = step;
    } else {
        const int G = a.G;
        if (touched) {
            o = rank;
            round = rank / G;
            slot = (round % 2) * G + rank % G;
            copy = !(round < 2 && s_occ[slot] == tid);
            s_last[rank] = tid;                            // expert by rank
        }
        __syncthreads();
        // the slot's occupant after the forward: the last touched expert that used it, else the
        // old one unless it was touched (and so moved or recopied elsewhere)
        if (tid < S) {
            int nw;
            if (tid < 2 * G && tid < U) {   // used first by rank tid, then every 2G ranks
                const int q = tid + ((U - 1 - tid) / (2 * G)) * 2 * G;
                nw = s_last[q];
                b.last_use[tid] = step;
            } else {
                const int pre = s_occ[tid];
                nw = (pre >= 0 && a.cnt[pre] > 0) ? -1 : pre;
            }
            s_use[tid] = (uint32_t)nw;
        }
        __syncthreads();
        if (tid < E && pre_slot >= 0 && (int)s_use[pre_slot] != tid) b.slot_of[tid] = -1;
        __syncthreads();
        if (tid < S) {
            const int nw = (int)s_use[tid];
            b.expert_in[tid] = nw;
            if (nw >= 0) b.slot_of[nw] = tid;
        }
    }

    // Round-ordered tiles and copies. Order index o: cache forward, resident experts then the
    // others, each in expert order; transient forward, the touched rank. Rounds are contiguous
    // runs of o.
    if (o >= 0) {   // s_aux is free again: the last victim read came before the last barrier
        s_order[o] = tid;
        s_oslot[o] = slot;
        s_oround[o] = round;
        s_aux[o] = copy;
    }
    __syncthreads();
    const int cp_flag_at_o = tid < U ? s_aux[tid] : 0;
    const int g = tid < U ? s_order[tid] : 0;
    const int cg = tid < U ? a.cnt[g] : 0;
    const int ts = (cg + a.ntile - 1) / a.ntile, tl = (cg + 2 * a.ntile - 1) / (2 * a.ntile);
    int TS, TL, NC;
    const int xs = block_exclusive_scan(ts, scan_smem, &TS);
    const int xl = block_exclusive_scan(tl, scan_smem, &TL);
    const int xc = block_exclusive_scan(cp_flag_at_o, scan_smem, &NC);
    const int rr = tid < U ? s_oround[tid] : -1;
    if (tid < U && (tid == 0 || s_oround[tid - 1] != rr)) {
        s_rs[rr] = xs;
        s_ls[rr] = xl;
        s_cs[rr] = xc;
    }
    __syncthreads();
    if (tid < U && (tid == U - 1 || s_oround[tid + 1] != rr)) {   // the round's last member
        b.counts[2 * rr] = xs + ts - s_rs[rr];
        b.counts[2 * rr + 1] = xl + tl - s_ls[rr];
        b.ncopy[rr] = xc + cp_flag_at_o - s_cs[rr];
        if (rr == 0) {
            s_sh_small = xs + ts;   // the shared expert's tiles follow round 0's
            s_sh_large = xl + tl;
        }
    }
    __syncthreads();
    if (tid < U) {
        const int sl = s_oslot[tid], base = a.off[g];
        int2 *rs = b.rec_small + (size_t)rr * b.nm + (xs - s_rs[rr]);
        for (int i = 0; i < ts; ++i) {
            const int n = min(a.ntile, cg - i * a.ntile);
            rs[i] = make_int2(base + i * a.ntile, sl | (n << 16));
        }
        int2 *rl = b.rec_large + (size_t)rr * b.nm + (xl - s_ls[rr]);
        for (int i = 0; i < tl; ++i) {
            const int n = min(2 * a.ntile, cg - i * 2 * a.ntile);
            rl[i] = make_int2(base + i * 2 * a.ntile, sl | (n << 16));
        }
        if (cp_flag_at_o) b.copies[(size_t)rr * S + (xc - s_cs[rr])] = make_int2(g, sl);
    }
    // the shared expert (group E) closes round 0
    const int csh = a.cnt[E];
    const int shs = (csh + a.ntile - 1) / a.ntile, shl = (csh + 2 * a.ntile - 1) / (2 * a.ntile);
    for (int i = tid; i < shs; i += kPlanThreads)
        b.rec_small[s_sh_small + i] = make_int2(a.off[E] + i * a.ntile, E | (min(a.ntile, csh - i * a.ntile) << 16));
    for (int i = tid; i < shl; i += kPlanThreads)
        b.rec_large[s_sh_large + i] =
            make_int2(a.off[E] + i * 2 * a.ntile, E | (min(2 * a.ntile, csh - i * 2 * a.ntile) << 16));
    if (tid == 0) {
        b.counts[0] += shs;
        b.counts[1] += shl;
        b.stats[0] = step;
        b.stats[1] += U - NC;
        b.stats[2] += NC;
    }
}

struct RefillArgs {
    const int2 *copies;
    const int32_t *ncopy;
    const uint8_t *src0, *src1, *src2, *src3;
    uint8_t *dst0, *dst1, *dst2, *dst3;
    uint64_t seg0, seg1, seg2, seg3;            // bytes per expert of each array (multiples of 16)
    uint64_t ch0, ch1, ch2;                     // cumulative 4 KB chunk counts of arrays 0..2
    uint64_t chunks;                            // 4 KB chunks per expert
    int E, S;
    int *err;
};

constexpr int kChunk = 4096;                    // bytes one warp moves per work item
constexpr int kRefillThreads = 1024;

// Each warp copies 4 KB chunks: eight 16-byte loads per lane in flight, then the stores. The
// source is read with plain loads (mapped host memory is device-accessible), the slot written
// with plain stores.
__global__ void __launch_bounds__(kRefillThreads) bank_refill(RefillArgs a) {
    const int n = *a.ncopy;
    const int lane = threadIdx.x & 31;
    const uint64_t warps = (uint64_t)gridDim.x * (kRefillThreads / 32);
    const uint64_t items = (uint64_t)n * a.chunks;
    for (uint64_t w = (uint64_t)blockIdx.x * (kRefillThreads / 32) + (threadIdx.x >> 5); w < items; w += warps) {
        const uint64_t c = w / a.chunks, k = w % a.chunks;
        const int2 cp = a.copies[c];
        if ((unsigned)cp.x >= (unsigned)a.E || (unsigned)cp.y >= (unsigned)a.S) {
            if (lane == 0) atomicCAS(a.err, 0, kErrBankCopy);
            continue;
        }
        const int sg = k < a.ch0 ? 0 : k < a.ch1 ? 1 : k < a.ch2 ? 2 : 3;
        const uint64_t kk = k - (sg == 0 ? 0 : sg == 1 ? a.ch0 : sg == 2 ? a.ch1 : a.ch2);
        const uint64_t seg = sg == 0 ? a.seg0 : sg == 1 ? a.seg1 : sg == 2 ? a.seg2 : a.seg3;
        const uint8_t *src = (sg == 0 ? a.src0 : sg == 1 ? a.src1 : sg == 2 ? a.src2 : a.src3) + cp.x * seg;
        uint8_t *dst = (sg == 0 ? a.dst0 : sg == 1 ? a.dst1 : sg == 2 ? a.dst2 : a.dst3) + cp.y * seg;
        const uint64_t lo = kk * kChunk, hi = min(seg, lo + kChunk);
        uint4 v[kChunk / 512];
#pragma unroll
        for (int j = 0; j < kChunk / 512; ++j) {
            const uint64_t off = lo + (uint64_t)j * 512 + lane * 16;
            if (off < hi) v[j] = *reinterpret_cast<const uint4 *>(src + off);
        }
#pragma unroll
        for (int j = 0; j < kChunk / 512; ++j) {
            const uint64_t off = lo + (uint64_t)j * 512 + lane * 16;
            if (off < hi) *reinterpret_cast<uint4 *>(dst + off) = v[j];
        }
    }
}

}  // namespace

int launch_bank_plan(const BankDev &b, const int32_t *cnt, const int32_t *off, bool cache, int G, int R, int ntile,
                     int *err, cudaStream_t st) {
    PlanArgs a;
    a.b = b;
    a.cnt = cnt;
    a.off = off;
    a.cache = cache ? 1 : 0;
    a.G = G;
    a.R = R;
    a.ntile = ntile;
    a.err = err;
    launch_pdl(bank_plan, dim3(1), dim3(kPlanThreads), 0, st, a);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

int launch_bank_refill(const BankDev &b, int r, const ExpertSet &src, const ExpertSet &dst, const ExpertBytes &eb,
                       int blocks, int *err, cudaStream_t st) {
    RefillArgs a;
    a.copies = b.copies + (size_t)r * b.S;
    a.ncopy = b.ncopy + r;
    a.src0 = src.gu_codes;
    a.src1 = src.gu_scales;
    a.src2 = src.d_codes;
    a.src3 = src.d_scales;
    a.dst0 = const_cast<uint8_t *>(dst.gu_codes);
    a.dst1 = const_cast<uint8_t *>(dst.gu_scales);
    a.dst2 = const_cast<uint8_t *>(dst.d_codes);
    a.dst3 = const_cast<uint8_t *>(dst.d_scales);
    a.seg0 = eb.seg[0];
    a.seg1 = eb.seg[1];
    a.seg2 = eb.seg[2];
    a.seg3 = eb.seg[3];
    const uint64_t c0 = (eb.seg[0] + kChunk - 1) / kChunk, c1 = (eb.seg[1] + kChunk - 1) / kChunk,
                   c2 = (eb.seg[2] + kChunk - 1) / kChunk, c3 = (eb.seg[3] + kChunk - 1) / kChunk;
    a.ch0 = c0;
    a.ch1 = c0 + c1;
    a.ch2 = c0 + c1 + c2;
    a.chunks = c0 + c1 + c2 + c3;
    a.E = b.E;
    a.S = b.S;
    a.err = err;
    bank_refill<<<blocks, kRefillThreads, 0, st>>>(a);
    return cudaPeekAtLastError() == cudaSuccess ? 1 : -1;
}

}  // namespace colimoe
