// The split-KV pass over a paged cache: the kernel of decode_split.cuh with
// PG = true, built in a translation unit of its own so that it compiles in
// parallel with the contiguous variants (decode_fast.cu).
#include "decode_split.cuh"

namespace kattn {

cudaError_t launch_split_paged(const DecodeParams& p, const TmaMaps& maps, cudaStream_t stream) {
  if (p.R <= 8) return launch_modes<1, 1, true>(p, maps, stream);
  if (const int nrg = row_groups_for(p); nrg > 1) {      // rows in groups of 8, a CTA each
    DecodeParams pr = p;
    pr.row_groups = nrg;
    return launch_modes<1, 1, true>(pr, maps, stream);
  }
  if (p.R <= 16) return launch_modes<2, 1, true>(p, maps, stream);
  if (p.R <= 32) return launch_split_tc(p, maps, stream);   // P.V on tcgen05 (decode_tc.cu)
  if (p.R <= 48) return launch_modes<3, 2, true>(p, maps, stream);
  return launch_modes<4, 2, true>(p, maps, stream);
}

}  // namespace kattn
