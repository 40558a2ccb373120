// status_slots.h -- per-plan device status words.
//
// Every kernel latches the bits of a bounded wait that gave up into the status
// word its plan hands it.  A plan takes its own word from a fixed device array
// (no allocation) so that conv_plan_device_status can report one plan's
// failures in the order of one stream; when all words are taken a plan shares
// the library-wide word that conv_device_status reads.
#pragma once

#include <cuda_runtime.h>

#include "../../include/conv.h"

namespace convgb {

// Take a free word on `device` and clear it (a device memset on the default
// stream).  On success *word is its device address and *slot its index; with
// none free, *slot = -1 and *word is the shared word.  Returns the first CUDA
// error met.
cudaError_t acquire_status_word(int device, unsigned** word, int* slot);

// Give a word back (slot -1: nothing to do).
void release_status_word(int device, int slot);

// Read and clear `word` in the order of `stream` (after the work queued on it), with
// `device` current: *code receives its bits.  CONV_ERR_TIMEOUT when any is set,
// CONV_ERR_INVALID_ARG for another current device, CONV_ERR_CUDA if a copy fails.
conv_status read_status_word(int device, unsigned* word, void* stream, int* code);

}  // namespace convgb
