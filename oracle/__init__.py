"""CPU oracle of the Dory looped nGPT token forward (test infrastructure only).

Only the tests, the package entry point's smoke check and the benchmark's CPU
baseline may import this package; the CUDA library never does.
"""
from .dory_oracle import DoryOracle, SeqState, Slot  # noqa: F401
