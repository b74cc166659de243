// anvil_schedule.h -- host-side phase table and item order of the cascade kernel.
#pragma once

#include "../../include/anvil.h"
#include "anvil_internal.h"

namespace anvil {

typedef anvil_map anvil_map_coef;

// Tiles of one matrix of bank b in a phase of op `op`.
int phase_tiles(const CascadeBank& b, int op);
// Fills cp->phase[] / cp->nphases for nmaps spectral maps (cp->bank[] and nbanks set).
void build_phases(CascadeParams* cp, const anvil_map_coef* maps, int nmaps);
// Phase by phase, banks in order, whole banks per run; phase_run (optional, nphases + 1
// entries) receives each phase's first run.
void order_phase_major(CascadeParams* cp, int* phase_run);

}  // namespace anvil
