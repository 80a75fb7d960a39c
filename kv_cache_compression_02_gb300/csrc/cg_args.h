// cg_args.h -- host-side validation of the (dims, params) pair that every
// entry point of libcachegen.so takes: the container and tables geometry
// (cg_layout.cuh) plus finite, positive level bases and layer multipliers.
// The decode entry points with and without a workspace share it, so they
// accept and reject exactly the same arguments.
#pragma once

#include <cmath>

#include "cachegen.h"
#include "cg_layout.cuh"

namespace cg {

inline bool layout_of(const cg_dims *dm, const cg_params *pr, Layout &lo) {
  if (!dm || !pr || dm->reserved != 0) return false;
  if (!make_layout(lo, dm->L, dm->H, dm->d, dm->C, dm->G, dm->S, pr->alphabet_radius, pr->n_levels))
    return false;
  for (int i = 0; i < pr->n_levels; i++)
    if (!std::isfinite(pr->level_base[i]) || !(pr->level_base[i] > 0.0f)) return false;
  if (pr->layer_mult)
    for (int i = 0; i < 2 * dm->L; i++)
      if (!std::isfinite(pr->layer_mult[i]) || !(pr->layer_mult[i] > 0.0f)) return false;
  return true;
}

}  // namespace cg
