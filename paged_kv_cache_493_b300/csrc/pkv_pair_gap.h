// pkv_pair_gap.h -- what a piece boundary costs in the split-K decode's
// stream-K plan (DecodeArgs::pair_gap), per entry point.
//
// The decode cuts the batch's chunks into equal slices of cost; a pair of n
// chunks costs pair_gap + n.  A block crossing more pairs than the others
// ends last unless each boundary is charged.  Set by measurement on B300:
// qwen_decode_b128's bf16 step is flat in it (62.4 us at 0, 62.1 at 1); its
// INT8 decode, whose 64-token chunks make a boundary cost more next to a
// chunk, goes from 53.2 us at 0 to 49.5 at 1 (50.9 at 2); the cascade's
// private parts are a few chunks per pair, and prefix_decode_b64 is best at
// 2 (31.6-32.8 us, against 32.7-32.9 at 0 and 1, 34.4 at 4).
#pragma once

namespace pkv {

constexpr int kPairGapDecode = 1;   // bf16 decode, fused store + decode, allocation-free decode
constexpr int kPairGapInt8 = 1;     // INT8 decode
constexpr int kPairGapCascade = 2;  // cascade decode's private parts

}  // namespace pkv
