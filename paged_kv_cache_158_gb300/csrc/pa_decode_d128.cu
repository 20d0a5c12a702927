#define PA_D 128
#include "pa_decode_inst.inc"
