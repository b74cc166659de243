// anvil_schedule.cu -- the host-side phase table and item order of the cascade kernel
// (anvil_gemm.cu).  The phases are those of the page "modded-nanogpt
// track_1_short/optim/anvil.py", anvil_cascade, for every bank: the first Gram (on X_raw,
// divided by d^2), then per spectral map the Gram (after the first map), B = bA + cA^2 and
// the X-update (the normalisation X / d runs before, in its own streaming kernel).  The
// order is a list of runs (anvil_internal.h).
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
    auto add = [&](int op, int ma, int mb, int min, int mout, float a, float b, float c) {
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
            ph.need_chain[q] = chain_total[q];
            chain_total[q] += SIGNALS_PER_TILE * static_cast<unsigned>(phase_tiles(cp->bank[q], op));
        }
    };
    // map k reads Y[(k+1)%2] and writes Y[k%2] (out for the last map)
    add(OP_GRAM_NORM, TM_YK0, TM_YK0, -1, TM_A, 0.f, 0.f, 0.f);
    for (int k = 0; k < nmaps; ++k) {
        const int cur = (k + 1) & 1;
        const bool last = k == nmaps - 1;
        if (k > 0) add(OP_GRAM, TM_YK0 + cur, TM_YK0 + cur, -1, TM_A, maps[k].a, maps[k].b, maps[k].c);
        add(OP_SQPOLY, TM_A, TM_A, TM_A, TM_B, maps[k].a, maps[k].b, maps[k].c);
        add(last ? OP_XUPDATE_OUT : OP_XUPDATE, TM_B, TM_YN0 + cur, TM_YK0 + cur,
            last ? TM_OUT : TM_YK0 + (cur ^ 1), maps[k].a, maps[k].b, maps[k].c);
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

}  // namespace anvil
