"""CPU oracle of the DFlash drafting step -- TEST INFRASTRUCTURE ONLY.

Importable only from the tests, the smoke check and the benchmark's CPU
baseline leg. The product library never imports, links or executes it.
"""
from . import dflash_ref, spec_loop  # noqa: F401
from .dflash_ref import (Cfg, argmax_lowest, attention, ctx_fuse, ctx_kv,  # noqa: F401
                         draft_block, rms_norm, rope, verify_accept)
