// merkle.h -- the block size of the Merkle passes, shared by the kernel (k_small.cu) and the
// workspace layout (repstep.cu).
#pragma once

#include <cstdint>

namespace repstep {

constexpr uint32_t kMerkleBlock = 1024;   // digests per block of a Merkle pass

}  // namespace repstep
