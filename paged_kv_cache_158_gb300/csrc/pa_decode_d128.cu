#define PA_D 128
#define PA_F8 0
#include "pa_decode_inst.inc"
