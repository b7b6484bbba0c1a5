"""CPU oracle of the drafting-round tree builder (test infrastructure, see oracle.cpp)."""
