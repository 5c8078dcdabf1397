// spec_device.cuh -- device code of the GB300 verify kernels (sm_103a).
//
// Verification runs two kernels per call. The stream kernel cuts the call's logits into units
// (one warp's share of one row: up to 32 lanes x 8 x 16-byte vectors = 4 KB of the row's
// 16-byte aligned interior), reads every unit exactly once with coalesced, L1-bypassing 128-bit
// loads and reduces it to one 8-byte partial: (max, sum of exp2((l - max) * log2(e)/T)) for
// softmax statistics, or (max value, lowest index) for greedy argmax. The finishing kernel, a
// programmatic dependent launch, combines the partials of each batch row and produces the
// outputs:
//
//   chain, T > 0  acceptance of every draft with one warp ballot, then the correction / bonus
//                 draw: an inverse CDF over max(0, p_n - q_n) (or p_gamma) over the one target
//                 and draft row the step stopped at, re-read from L2 and split over the CTAs
//                 of a thread-block cluster (a bonus draw from the unit partials alone when it
//                 can); rows of a single unit finish in one warp per batch row;
//   chain, T = 0  argmax comparison of every draft token, then the greedy correction token;
//   tree          accepted set and depths of all nodes, deepest node, path and bonus token;
//   tree, T > 0   the walk from the root by per-sibling rejection sampling (one CTA per tree).
//
// The probability helper holds each row in the registers of a cluster of CTAs (one kernel, one
// read and one write); top-n candidates follow the stream / finish pattern; the tree mask is
// one CTA per tree.
//
// No CTA ever waits for another CTA of its own grid except through the hardware cluster
// barrier. Data written by other CTAs is read with ld.global.cg (L2), never through L1.
//
// Parts, in dependency order:
//   spec_common.cuh   constants, parameters, element access, row geometry, unit reductions
//   spec_draw.cuh     the inverse-CDF draw over residual segments
//   spec_finish.cuh   combining partials, acceptance, emitting, greedy chains, trees, cluster
//                     draws
//   spec_kernels.cuh  the verification and probability kernels
//   spec_tree_sample.cuh  stochastic tree verification: the walk by per-sibling rejection
//   spec_helpers.cuh  top-n candidates and the tree-attention mask
#pragma once

#include "spec_common.cuh"
#include "spec_draw.cuh"
#include "spec_finish.cuh"
#include "spec_kernels.cuh"
#include "spec_tree_sample.cuh"
#include "spec_helpers.cuh"
