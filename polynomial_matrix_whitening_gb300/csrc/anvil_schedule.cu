// anvil_schedule.cu -- the host-side phase table and item order of the cascade kernel
// (anvil_gemm.cu).  The phases are those of the page "modded-nanogpt
// track_1_short/optim/anvil.py", anvil_cascade, for every bank: the first Gram (on X_raw,
// divided by d^2), the normalisation X / d, then per spectral map the Gram (after the
// first map), B = bA + cA^2 and the X-update.  The order is a list of runs (anvil_internal.h).
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "anvil_internal.h"
#include "anvil_schedule.h"

namespace anvil {

static bool sym_op(int op) { return op == OP_GRAM || op == OP_GRAM_NORM || op == OP_SQPOLY; }

int phase_tiles(const CascadeBank& b, int op) {
    return sym_op(op) ? b.T * (b.T + 1) / 2 : b.T * b.ntl;
}

void build_phases(CascadeParams* cp, const anvil_map_coef* maps, int nmaps) {
    unsigned chain_total[MAX_BANKS] = {0};  // chain signals per matrix of each bank so far
    int nph = 0;
    auto add = [&](int op, int ma, int mb, int min, int mout, float a, float b, float c, bool after_norm) {
        CascadePhase& ph = cp->phase[nph++];
        ph.op = op;
        ph.map_a = ma;
        ph.map_b = mb;
        ph.map_in = min;
        ph.map_out = mout;
        // the symmetric operands: A (both operands of A A) and B (the X-update's left factor)
        ph.map_a_t = ma == TM_A ? TM_AN : ma == TM_B ? TM_BN : -1;
        ph.map_b_t = mb == TM_A ? TM_AN : -1;
        ph.a = a;
        ph.b = b;
        ph.c = c;
        for (int q = 0; q < cp->nbanks; ++q) {
            const CascadeBank& cb = cp->bank[q];
            if (op == OP_NORMALIZE) {
                ph.need_chain[q] = 0;
                ph.need_norm[q] = 0;
            } else {
                ph.need_chain[q] = chain_total[q];
                ph.need_norm[q] = after_norm ? SIGNALS_PER_TILE * static_cast<unsigned>(cb.T * cb.ntl) : 0u;
                chain_total[q] += SIGNALS_PER_TILE * static_cast<unsigned>(phase_tiles(cb, op));
            }
        }
    };
    // map k reads Y[(k+1)%2] and writes Y[k%2] (out for the last map)
    add(OP_GRAM_NORM, TM_YK0, TM_YK0, -1, TM_A, 0.f, 0.f, 0.f, false);
    add(OP_NORMALIZE, -1, -1, TM_YK0, TM_YK1, 0.f, 0.f, 0.f, false);
    for (int k = 0; k < nmaps; ++k) {
        const int cur = (k + 1) & 1;
        const bool last = k == nmaps - 1;
        if (k > 0) add(OP_GRAM, TM_YK0 + cur, TM_YK0 + cur, -1, TM_A, maps[k].a, maps[k].b, maps[k].c, false);
        add(OP_SQPOLY, TM_A, TM_A, TM_A, TM_B, maps[k].a, maps[k].b, maps[k].c, false);
        add(last ? OP_XUPDATE_OUT : OP_XUPDATE, TM_B, TM_YN0 + cur, TM_YK0 + cur,
            last ? TM_OUT : TM_YK0 + (cur ^ 1), maps[k].a, maps[k].b, maps[k].c, k == 0);
    }
    cp->nphases = nph;
}

// Phase by phase, banks in their order (heaviest first), all matrices of a bank in one run.
// phase_run[p] receives the first run of phase p (phase_run[nphases] = nruns).
void order_phase_major(CascadeParams* cp, int* phase_run) {
    int items = 0, nr = 0;
    for (int p = 0; p < cp->nphases; ++p) {
        if (phase_run) phase_run[p] = nr;
        for (int q = 0; q < cp->nbanks; ++q) {
            const CascadeBank& b = cp->bank[q];
            CascadeRun& r = cp->run[nr++];
            r.begin = items;
            r.phase = static_cast<uint8_t>(p);
            r.bank = static_cast<uint8_t>(q);
            r.mat0 = 0;
            r.nmat = static_cast<uint32_t>(b.g);
            items += b.g * phase_tiles(b, cp->phase[p].op);
        }
    }
    if (phase_run) phase_run[cp->nphases] = nr;
    cp->nruns = nr;
    cp->run[nr].begin = items;
}

// Phase by phase as order_phase_major, except that the normalisation's items, which use
// no tensor cores, are spread matrix by matrix over the product phases that come before
// the first X-update (the first Gram and the first B = bA + cA^2, which do not read the
// normalised X): a pair's epilogue warps then divide tiles while its MMAs run.  The
// spread keeps the normalisation's share of the emitted cost equal to the products'
// share; costs are k-blocks of 64 for a product tile and kNormCost for a normalisation
// tile.
void order_normalize_interleaved(CascadeParams* cp) {
    const double kNormCost = 14.0;
    // one run per matrix and phase before the first X-update at most: past the run
    // table's capacity (or the 16-bit matrix index), the plain phase-major order
    long long mats = 0;
    int gmax = 0;
    for (int q = 0; q < cp->nbanks; ++q) {
        mats += cp->bank[q].g;
        gmax = std::max(gmax, cp->bank[q].g);
    }
    if (3 * mats + static_cast<long long>(cp->nphases) * cp->nbanks > MAX_RUNS || gmax > 65535) {
        order_phase_major(cp, nullptr);
        return;
    }
    int first_x = cp->nphases;  // the first X-update phase
    int pn = -1;                // the normalisation phase
    for (int p = 0; p < cp->nphases; ++p) {
        const int op = cp->phase[p].op;
        if (op == OP_NORMALIZE && pn < 0) pn = p;
        if ((op == OP_XUPDATE || op == OP_XUPDATE_OUT) && first_x == cp->nphases) first_x = p;
    }
    struct Seg {
        int phase, bank, mat;
        double cost;
    };
    std::vector<Seg> prod, norm, order;
    for (int p = 0; p < first_x; ++p)
        for (int q = 0; q < cp->nbanks; ++q) {
            const CascadeBank& b = cp->bank[q];
            const int op = cp->phase[p].op;
            const double per = op == OP_NORMALIZE ? kNormCost
                                                  : ((op == OP_GRAM || op == OP_GRAM_NORM) ? b.L_pad : b.s_pad) / 64.0;
            for (int i = 0; i < b.g; ++i)
                (p == pn ? norm : prod).push_back({p, q, i, per * phase_tiles(b, op)});
        }
    double tot_p = 0.0, tot_n = 0.0;
    for (const Seg& x : prod) tot_p += x.cost;
    for (const Seg& x : norm) tot_n += x.cost;
    size_t ip = 0, in = 0;
    double cum_p = 0.0, cum_n = 0.0;
    while (ip < prod.size() || in < norm.size()) {
        const bool take_n = in < norm.size() && (ip == prod.size() || cum_n * tot_p <= cum_p * tot_n);
        if (take_n) {
            cum_n += norm[in].cost;
            order.push_back(norm[in++]);
        } else {
            cum_p += prod[ip].cost;
            order.push_back(prod[ip++]);
        }
    }
    for (int p = first_x; p < cp->nphases; ++p)
        for (int q = 0; q < cp->nbanks; ++q) order.push_back({p, q, -1, 0.0});
    int items = 0, nr = 0;
    for (const Seg& x : order) {
        const CascadeBank& b = cp->bank[x.bank];
        const int tiles = phase_tiles(b, cp->phase[x.phase].op);
        const int nmat = x.mat < 0 ? b.g : 1;
        if (x.mat >= 0 && nr > 0) {
            CascadeRun& last = cp->run[nr - 1];
            if (last.phase == x.phase && last.bank == x.bank && static_cast<int>(last.mat0 + last.nmat) == x.mat) {
                last.nmat += 1;
                items += tiles;
                continue;
            }
        }
        CascadeRun& r = cp->run[nr++];
        r.begin = items;
        r.phase = static_cast<uint8_t>(x.phase);
        r.bank = static_cast<uint8_t>(x.bank);
        r.mat0 = static_cast<uint16_t>(x.mat < 0 ? 0 : x.mat);
        r.nmat = static_cast<uint32_t>(nmat);
        items += nmat * tiles;
    }
    cp->nruns = nr;
    cp->run[nr].begin = items;
}

}  // namespace anvil
