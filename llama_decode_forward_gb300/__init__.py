"""Batch-1 Llama decode forward pass on one GB300 (sm_103a).

The computation lives in the CUDA library libllmdecode (csrc/, C ABI in
include/llm.h); ``binding`` marshals arguments to it.  Importing the package
builds the library if needed and fails if it cannot be built or loaded.
"""
from .binding import *  # noqa: F401,F403
from .binding import Decoder, DeviceWeights, LlmError, LIBRARY_PATH, declared_symbols  # noqa: F401
